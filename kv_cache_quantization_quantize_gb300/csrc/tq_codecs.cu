// Comparison KV codecs of the TurboQuant-vLLM overview (§核心技术解析): KIVI 2-bit (keys per channel,
// values per token, asymmetric scale + zero point) and Bonsai 1-bit (sign codes with one fp16 scale per
// 128 channels). Both are streaming, HBM-bound kernels: every element is read once and its code
// written once; there is no contraction, so no tensor-core work.
//
// Readings (the overview names the schemes, not their parameters; these reproduce the KV sizes of its
// table in §性能表现与实测数据):
//   KIVI: groups of 16 (16 tokens of one key channel; 16 channels of one value token); zero z = fp16(min),
//         scale s = fp16((max - min) / 3); code = clamp(rint((x - z) * r), 0, 3) with r = 1/s, every
//         step in fp32 round-to-nearest-even (code 0 where s = 0); x_hat = z + code * s.
//   Bonsai: bit = (x >= 0); scale = fp16(mean |x|) over 128 consecutive channels; x_hat = +-scale.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kCodecThreads = 256;
constexpr int kKiviGroup = 16;
constexpr int kBonsaiGroup = 128;
// Adding 1.5 * 2^23 to a float in [0, 4) leaves rint(x) (round half to even) in the low mantissa bits.
constexpr float kRoundMagic = 12582912.0f;
constexpr uint32_t kMagicBits = 0x4B400000u;
// Horner packing of sixteen (kMagicBits + code) words, base 4, adds kMagicBits * (4^16 - 1) / 3.
constexpr uint32_t kMagicPack16 = kMagicBits * 0x55555555u;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Group parameters from the group's min and max: fp16 bits of (scale, zero) and the fp32 values used
// to code (zero, reciprocal of scale; r = 0 when the scale is 0, so every code is 0).
struct KiviGroup {
  float z, r;
  uint16_t sh, zh;
};

__device__ __forceinline__ KiviGroup kivi_group(float lo, float hi) {
  KiviGroup g;
  const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 3.0f));
  const __half z16 = __float2half_rn(lo);
  const float s = __half2float(s16);
  g.z = __half2float(z16);
  g.r = s == 0.f ? 0.f : __frcp_rn(s);
  g.sh = __half_as_ushort(s16);
  g.zh = __half_as_ushort(z16);
  return g;
}

// kMagicBits + code for one element (code in 0..3).
__device__ __forceinline__ uint32_t kivi_code(float x, const KiviGroup& g) {
  const float v = fminf(fmaxf(__fmul_rn(__fsub_rn(x, g.z), g.r), 0.f), 3.f);
  return __float_as_uint(__fadd_rn(v, kRoundMagic));
}

struct KiviArgs {
  const uint32_t* k;   // bf16 pairs [T][C/2], C = n_heads * head_dim
  const uint4* v;      // bf16 octets [T][C/8]
  uint2* k_codes;      // [T/16][C] uint32, written as channel pairs
  uint32_t* k_scale;   // [T/16][C] fp16, written as channel pairs
  uint32_t* k_zero;
  uint32_t* v_codes;   // [T][C/16]
  uint16_t* v_scale;   // [T][C/16]
  uint16_t* v_zero;
  long long n_key_items;  // (T/16) * C/2 channel pairs
  long long n_val_groups;  // T * C/16 groups
  long long n_val_items;   // ceil(groups / 2): a value thread codes two groups
  int half_c;             // C/2
  int key_blocks;         // blocks [0, key_blocks) code keys, the rest code values
};

// Keys: one thread per (16-token group, channel pair). Sixteen coalesced 4-byte row loads, then both
// channels' codes, packed token t at bits 2t..2t+1.
__device__ __forceinline__ void kivi_key_item(const KiviArgs& a, long long item) {
  const long long g = item / a.half_c;
  const int j = (int)(item - g * a.half_c);
  const uint32_t* src = a.k + (size_t)g * kKiviGroup * a.half_c + j;
  uint32_t w[kKiviGroup];
#pragma unroll
  for (int t = 0; t < kKiviGroup; ++t) w[t] = __ldcs(src + (size_t)t * a.half_c);
  float lo0 = bf_lo(w[0]), hi0 = lo0, lo1 = bf_hi(w[0]), hi1 = lo1;
#pragma unroll
  for (int t = 1; t < kKiviGroup; ++t) {
    lo0 = fminf(lo0, bf_lo(w[t]));
    hi0 = fmaxf(hi0, bf_lo(w[t]));
    lo1 = fminf(lo1, bf_hi(w[t]));
    hi1 = fmaxf(hi1, bf_hi(w[t]));
  }
  const KiviGroup p0 = kivi_group(lo0, hi0), p1 = kivi_group(lo1, hi1);
  uint32_t c0 = 0, c1 = 0;
#pragma unroll
  for (int t = kKiviGroup - 1; t >= 0; --t) {
    c0 = c0 * 4u + kivi_code(bf_lo(w[t]), p0);
    c1 = c1 * 4u + kivi_code(bf_hi(w[t]), p1);
  }
  const size_t o = (size_t)g * a.half_c + j;
  __stcs(a.k_codes + o, make_uint2(c0 - kMagicPack16, c1 - kMagicPack16));
  __stcs(a.k_scale + o, (uint32_t)p0.sh | ((uint32_t)p1.sh << 16));
  __stcs(a.k_zero + o, (uint32_t)p0.zh | ((uint32_t)p1.zh << 16));
}

// Values: one thread per two (token, 16-channel) groups (64 bytes in flight); channel i at bits 2i..2i+1.
__device__ __forceinline__ void kivi_value_group(const KiviArgs& a, long long grp, const uint4& q0, const uint4& q1) {
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  float lo = bf_lo(w[0]), hi = lo;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a0 = bf_lo(w[i]), a1 = bf_hi(w[i]);
    lo = fminf(lo, fminf(a0, a1));
    hi = fmaxf(hi, fmaxf(a0, a1));
  }
  const KiviGroup p = kivi_group(lo, hi);
  uint32_t c = 0;
#pragma unroll
  for (int i = 7; i >= 0; --i) {
    c = c * 4u + kivi_code(bf_hi(w[i]), p);
    c = c * 4u + kivi_code(bf_lo(w[i]), p);
  }
  __stcs(a.v_codes + grp, c - kMagicPack16);
  __stcs(a.v_scale + grp, p.sh);
  __stcs(a.v_zero + grp, p.zh);
}

__device__ __forceinline__ void kivi_value_item(const KiviArgs& a, long long item) {
  const long long g0 = 2 * item;
  const bool two = g0 + 1 < a.n_val_groups;
  const uint4 q0 = __ldcs(a.v + 2 * g0), q1 = __ldcs(a.v + 2 * g0 + 1);
  uint4 q2 = make_uint4(0u, 0u, 0u, 0u), q3 = q2;
  if (two) {
    q2 = __ldcs(a.v + 2 * g0 + 2);
    q3 = __ldcs(a.v + 2 * g0 + 3);
  }
  kivi_value_group(a, g0, q0, q1);
  if (two) kivi_value_group(a, g0 + 1, q2, q3);
}

__global__ void __launch_bounds__(kCodecThreads) k_kivi2_quantize(const KiviArgs a) {
  if ((int)blockIdx.x < a.key_blocks) {
    const long long item = (long long)blockIdx.x * kCodecThreads + threadIdx.x;
    if (item < a.n_key_items) kivi_key_item(a, item);
  } else {
    const long long item = (long long)(blockIdx.x - a.key_blocks) * kCodecThreads + threadIdx.x;
    if (item < a.n_val_items) kivi_value_item(a, item);
  }
}

// x_hat of one code as bf16: zero + code * scale in fp32 (code * scale is exact), rounded to bf16.
__device__ __forceinline__ float kivi_level(uint32_t code, float s, float z) {
  return fmaf(__uint_as_float(kMagicBits | code) - kRoundMagic, s, z);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

struct KiviDeqArgs {
  const uint2* k_codes;
  const uint32_t* k_scale;
  const uint32_t* k_zero;
  const uint32_t* v_codes;
  const uint16_t* v_scale;
  const uint16_t* v_zero;
  uint32_t* k_out;  // bf16 pairs [T][C/2]
  uint4* v_out;     // bf16 octets [T][C/8]
  long long n_key_items, n_val_items;
  int half_c, key_blocks;
};

__global__ void __launch_bounds__(kCodecThreads) k_kivi2_dequantize(const KiviDeqArgs a) {
  if ((int)blockIdx.x < a.key_blocks) {
    const long long item = (long long)blockIdx.x * kCodecThreads + threadIdx.x;
    if (item >= a.n_key_items) return;
    const long long g = item / a.half_c;
    const int j = (int)(item - g * a.half_c);
    const size_t o = (size_t)g * a.half_c + j;
    const uint2 c = __ldcs(a.k_codes + o);
    const uint32_t sh = __ldcs(a.k_scale + o), zh = __ldcs(a.k_zero + o);
    const float s0 = __half2float(__ushort_as_half((uint16_t)sh)), s1 = __half2float(__ushort_as_half((uint16_t)(sh >> 16)));
    const float z0 = __half2float(__ushort_as_half((uint16_t)zh)), z1 = __half2float(__ushort_as_half((uint16_t)(zh >> 16)));
    uint32_t* dst = a.k_out + (size_t)g * kKiviGroup * a.half_c + j;
#pragma unroll
    for (int t = 0; t < kKiviGroup; ++t)
      __stcs(dst + (size_t)t * a.half_c,
             pack_bf16x2(kivi_level((c.x >> (2 * t)) & 3u, s0, z0), kivi_level((c.y >> (2 * t)) & 3u, s1, z1)));
  } else {
    const long long item = (long long)(blockIdx.x - a.key_blocks) * kCodecThreads + threadIdx.x;
    if (item >= a.n_val_items) return;
    const uint32_t c = __ldcs(a.v_codes + item);
    const float s = __half2float(__ushort_as_half(__ldcs(a.v_scale + item)));
    const float z = __half2float(__ushort_as_half(__ldcs(a.v_zero + item)));
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = pack_bf16x2(kivi_level((c >> (4 * i)) & 3u, s, z), kivi_level((c >> (4 * i + 2)) & 3u, s, z));
    __stcs(a.v_out + 2 * item, make_uint4(w[0], w[1], w[2], w[3]));
    __stcs(a.v_out + 2 * item + 1, make_uint4(w[4], w[5], w[6], w[7]));
  }
}

// Bonsai: a warp codes spans of 256 channels (two groups); lane l reads channels 8l..8l+7 of a span
// with one 16-byte load. Its eight sign bits form byte l % 4 of word l / 4 (channel 32w + b at bit b);
// the |x| sums of lanes 0-15 and 16-31 are the two groups' sums, reduced in a fixed butterfly order.
constexpr int kBonsaiSpansPerWarp = 4;

struct BonsaiArgs {
  const uint4* x[2];     // K, V: bf16 [rows][d] viewed as 16-byte octets (NULL = skip)
  uint32_t* bits[2];     // [rows][d/32]
  uint16_t* scale[2];    // [rows][d/128]
  long long n_groups;    // rows * d / 128 per tensor
  long long warps_per_tensor;
};

__global__ void __launch_bounds__(kCodecThreads) k_bonsai1_quantize(const BonsaiArgs a) {
  const long long gw = ((long long)blockIdx.x * kCodecThreads + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int which = gw >= a.warps_per_tensor ? 1 : 0;
  if (which && gw >= 2 * a.warps_per_tensor) return;  // whole warp exits together
  const long long w = gw - which * a.warps_per_tensor;
  const uint4* src = which ? a.x[1] : a.x[0];
  uint32_t* bits = which ? a.bits[1] : a.bits[0];
  uint16_t* scale = which ? a.scale[1] : a.scale[0];
  if (!src) return;
  const long long n_spans = (a.n_groups + 1) / 2;
  uint4 q[kBonsaiSpansPerWarp];
#pragma unroll
  for (int u = 0; u < kBonsaiSpansPerWarp; ++u) {
    const long long span = w * kBonsaiSpansPerWarp + u;
    const bool live = span < n_spans && (lane < 16 || 2 * span + 1 < a.n_groups);
    q[u] = live ? __ldcs(src + span * 32 + lane) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < kBonsaiSpansPerWarp; ++u) {
    const long long span = w * kBonsaiSpansPerWarp + u;
    if (span >= n_spans) break;  // uniform across the warp
    const uint32_t e[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
    float sum = 0.f;
    uint32_t byte = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float f0 = bf_lo(e[i]), f1 = bf_hi(e[i]);
      sum += fabsf(f0);
      sum += fabsf(f1);
      byte |= (f0 >= 0.f ? 1u : 0u) << (2 * i);
      byte |= (f1 >= 0.f ? 1u : 0u) << (2 * i + 1);
    }
    uint32_t word = byte << (8 * (lane & 3));
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, m);
    const long long grp = 2 * span + (lane >> 4);
    if (grp < a.n_groups) {
      if ((lane & 3) == 0) __stcs(bits + span * 8 + (lane >> 2), word);
      if ((lane & 15) == 0) __stcs(scale + grp, __half_as_ushort(__float2half_rn(sum * (1.0f / kBonsaiGroup))));
    }
  }
}

struct BonsaiDeqArgs {
  const uint32_t* bits[2];
  const uint16_t* scale[2];
  uint4* out[2];        // bf16 [rows][d]
  long long n_words;    // rows * d / 32 per tensor
};

// One thread per 8 channels (a byte of a code word): one 16-byte store, consecutive threads writing
// consecutive bytes of the output. +scale or -scale by bit.
__global__ void __launch_bounds__(kCodecThreads) k_bonsai1_dequantize(const BonsaiDeqArgs a) {
  long long item = (long long)blockIdx.x * kCodecThreads + threadIdx.x;
  const long long per_tensor = 4 * a.n_words;
  const int which = item >= per_tensor ? 1 : 0;
  item -= which * per_tensor;
  const uint32_t* bits = which ? a.bits[1] : a.bits[0];
  const uint16_t* scale = which ? a.scale[1] : a.scale[0];
  uint4* out = which ? a.out[1] : a.out[0];
  if (item >= per_tensor || !bits) return;
  const long long word = item >> 2;
  const uint32_t neg = ~__ldg(bits + word) >> (8 * (int)(item & 3));
  const uint32_t sb = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(
      __half2float(__ushort_as_half(__ldg(scale + word / (kBonsaiGroup / 32))))));
  const uint32_t ss = sb | (sb << 16);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = neg >> (2 * i);
    o[i] = ss | ((t << 15) & 0x8000u) | ((t << 30) & 0x80000000u);
  }
  __stcs(out + item, make_uint4(o[0], o[1], o[2], o[3]));
}

bool misaligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; }

long long blocks_for(long long items) { return (items + kCodecThreads - 1) / kCodecThreads; }

}  // namespace
}  // namespace tq

extern "C" size_t tq_codec_kv_bytes(int codec, int n_layers, int n_kv_heads, int head_dim, int64_t n_tokens) {
  if (n_layers < 1 || n_kv_heads < 1 || head_dim < 1 || n_tokens < 0) return 0;
  const size_t vectors = (size_t)n_layers * n_kv_heads * (size_t)n_tokens;  // per tensor (K or V)
  const size_t elems = vectors * head_dim;
  switch (codec) {
    case TQ_CODEC_FP16:
      return 2 * 2 * elems;
    case TQ_CODEC_KIVI2:  // 2-bit codes + fp16 scale and zero per 16 elements, for K and V
      if (head_dim % tq::kKiviGroup) return 0;
      return 2 * (elems / 4 + 4 * (elems / tq::kKiviGroup));
    case TQ_CODEC_BONSAI1:  // 1-bit codes + fp16 scale per 128 elements, for K and V
      if (head_dim % tq::kBonsaiGroup) return 0;
      return 2 * (elems / 8 + 2 * (elems / tq::kBonsaiGroup));
    case TQ_CODEC_TQ_K3V2:  // key record d/4 + d/8 + 4 bytes, value record d/4 + d/16 bytes
    case TQ_CODEC_TQ_K3V4: {  // value record d/2 + d/16 bytes
      if (head_dim % 32) return 0;
      const size_t key = head_dim / 4 + head_dim / 8 + 4;
      const size_t val = (codec == TQ_CODEC_TQ_K3V2 ? head_dim / 4 : head_dim / 2) + head_dim / 16;
      return vectors * (key + val);
    }
    default:
      return 0;
  }
}

extern "C" tq_status tq_kivi2_quantize(const void* k, const void* v, int n_tokens, int n_heads, int head_dim,
                                       uint32_t* k_codes, uint16_t* k_scale, uint16_t* k_zero, uint32_t* v_codes,
                                       uint16_t* v_scale, uint16_t* v_zero, tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_kivi2_quantize");
  using namespace tq;
  if (n_tokens < 0 || n_heads < 1 || head_dim < 16 || head_dim % kKiviGroup)
    return set_error(TQ_ERR_INVALID_ARG, "kivi2: n_tokens >= 0, n_heads >= 1, head_dim a multiple of 16 >= 16");
  if (k && n_tokens % kKiviGroup)
    return set_error(TQ_ERR_INVALID_ARG, "kivi2: keys need a multiple of 16 tokens (per-channel groups of 16)");
  if (k && (!k_codes || !k_scale || !k_zero)) return set_error(TQ_ERR_INVALID_ARG, "kivi2: NULL key output");
  if (v && (!v_codes || !v_scale || !v_zero)) return set_error(TQ_ERR_INVALID_ARG, "kivi2: NULL value output");
  if (misaligned(k, 16) || misaligned(v, 16) || misaligned(k_codes, 8) || misaligned(k_scale, 4) ||
      misaligned(k_zero, 4) || misaligned(v_codes, 4) || misaligned(v_scale, 2) || misaligned(v_zero, 2))
    return set_error(TQ_ERR_INVALID_ARG, "kivi2: k/v 16-byte, k_codes 8-byte, k_scale/k_zero/v_codes 4-byte aligned");
  const long long C = (long long)n_heads * head_dim;
  KiviArgs a{};
  a.k = static_cast<const uint32_t*>(k);
  a.v = static_cast<const uint4*>(v);
  a.k_codes = reinterpret_cast<uint2*>(k_codes);
  a.k_scale = reinterpret_cast<uint32_t*>(k_scale);
  a.k_zero = reinterpret_cast<uint32_t*>(k_zero);
  a.v_codes = v_codes;
  a.v_scale = v_scale;
  a.v_zero = v_zero;
  a.half_c = (int)(C / 2);
  a.n_key_items = k ? (long long)(n_tokens / kKiviGroup) * (C / 2) : 0;
  a.n_val_groups = v ? (long long)n_tokens * (C / kKiviGroup) : 0;
  a.n_val_items = (a.n_val_groups + 1) / 2;
  if (C / 2 > INT32_MAX) return set_error(TQ_ERR_INVALID_ARG, "kivi2: n_heads * head_dim too large");
  const long long kb = blocks_for(a.n_key_items), vb = blocks_for(a.n_val_items);
  if (kb + vb == 0) return set_error(TQ_OK, "");
  if (kb + vb > INT32_MAX) return set_error(TQ_ERR_INVALID_ARG, "kivi2: too many elements for one launch");
  a.key_blocks = (int)kb;
  k_kivi2_quantize<<<(unsigned)(kb + vb), kCodecThreads, 0, (cudaStream_t)stream>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(TQ_ERR_CUDA, cudaGetErrorString(e));
  return set_error(TQ_OK, "");
}

extern "C" tq_status tq_kivi2_dequantize(const uint32_t* k_codes, const uint16_t* k_scale, const uint16_t* k_zero,
                                         const uint32_t* v_codes, const uint16_t* v_scale, const uint16_t* v_zero,
                                         int n_tokens, int n_heads, int head_dim, void* k_out, void* v_out,
                                         tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_kivi2_dequantize");
  using namespace tq;
  if (n_tokens < 0 || n_heads < 1 || head_dim < 16 || head_dim % kKiviGroup)
    return set_error(TQ_ERR_INVALID_ARG, "kivi2: n_tokens >= 0, n_heads >= 1, head_dim a multiple of 16 >= 16");
  if (k_out && n_tokens % kKiviGroup)
    return set_error(TQ_ERR_INVALID_ARG, "kivi2: keys need a multiple of 16 tokens (per-channel groups of 16)");
  if (k_out && (!k_codes || !k_scale || !k_zero)) return set_error(TQ_ERR_INVALID_ARG, "kivi2: NULL key input");
  if (v_out && (!v_codes || !v_scale || !v_zero)) return set_error(TQ_ERR_INVALID_ARG, "kivi2: NULL value input");
  if (misaligned(k_out, 16) || misaligned(v_out, 16) || misaligned(k_codes, 8) || misaligned(k_scale, 4) ||
      misaligned(k_zero, 4) || misaligned(v_codes, 4) || misaligned(v_scale, 2) || misaligned(v_zero, 2))
    return set_error(TQ_ERR_INVALID_ARG, "kivi2: outputs 16-byte, k_codes 8-byte, k_scale/k_zero/v_codes 4-byte aligned");
  const long long C = (long long)n_heads * head_dim;
  if (C / 2 > INT32_MAX) return set_error(TQ_ERR_INVALID_ARG, "kivi2: n_heads * head_dim too large");
  KiviDeqArgs a{};
  a.k_codes = reinterpret_cast<const uint2*>(k_codes);
  a.k_scale = reinterpret_cast<const uint32_t*>(k_scale);
  a.k_zero = reinterpret_cast<const uint32_t*>(k_zero);
  a.v_codes = v_codes;
  a.v_scale = v_scale;
  a.v_zero = v_zero;
  a.k_out = static_cast<uint32_t*>(k_out);
  a.v_out = static_cast<uint4*>(v_out);
  a.half_c = (int)(C / 2);
  a.n_key_items = k_out ? (long long)(n_tokens / kKiviGroup) * (C / 2) : 0;
  a.n_val_items = v_out ? (long long)n_tokens * (C / kKiviGroup) : 0;
  const long long kb = blocks_for(a.n_key_items), vb = blocks_for(a.n_val_items);
  if (kb + vb == 0) return set_error(TQ_OK, "");
  if (kb + vb > INT32_MAX) return set_error(TQ_ERR_INVALID_ARG, "kivi2: too many elements for one launch");
  a.key_blocks = (int)kb;
  k_kivi2_dequantize<<<(unsigned)(kb + vb), kCodecThreads, 0, (cudaStream_t)stream>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(TQ_ERR_CUDA, cudaGetErrorString(e));
  return set_error(TQ_OK, "");
}

extern "C" tq_status tq_bonsai1_quantize(const void* k, const void* v, int64_t n_rows, int head_dim, uint32_t* k_bits,
                                         uint16_t* k_scale, uint32_t* v_bits, uint16_t* v_scale, tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_bonsai1_quantize");
  using namespace tq;
  if (n_rows < 0 || head_dim < kBonsaiGroup || head_dim % kBonsaiGroup)
    return set_error(TQ_ERR_INVALID_ARG, "bonsai1: n_rows >= 0 and head_dim a multiple of 128");
  if ((k && (!k_bits || !k_scale)) || (v && (!v_bits || !v_scale)))
    return set_error(TQ_ERR_INVALID_ARG, "bonsai1: NULL output");
  if (misaligned(k, 16) || misaligned(v, 16) || misaligned(k_bits, 4) || misaligned(v_bits, 4) ||
      misaligned(k_scale, 2) || misaligned(v_scale, 2))
    return set_error(TQ_ERR_INVALID_ARG, "bonsai1: k/v 16-byte and bits 4-byte aligned");
  BonsaiArgs a{};
  a.x[0] = static_cast<const uint4*>(k);
  a.x[1] = static_cast<const uint4*>(v);
  a.bits[0] = k_bits;
  a.bits[1] = v_bits;
  a.scale[0] = k_scale;
  a.scale[1] = v_scale;
  a.n_groups = n_rows * (head_dim / kBonsaiGroup);
  const long long spans = (a.n_groups + 1) / 2;
  a.warps_per_tensor = (spans + kBonsaiSpansPerWarp - 1) / kBonsaiSpansPerWarp;
  if ((!k && !v) || a.n_groups == 0) return set_error(TQ_OK, "");
  const long long blocks = (2 * a.warps_per_tensor * 32 + kCodecThreads - 1) / kCodecThreads;
  if (blocks > INT32_MAX) return set_error(TQ_ERR_INVALID_ARG, "bonsai1: too many rows for one launch");
  k_bonsai1_quantize<<<(unsigned)blocks, kCodecThreads, 0, (cudaStream_t)stream>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(TQ_ERR_CUDA, cudaGetErrorString(e));
  return set_error(TQ_OK, "");
}

extern "C" tq_status tq_bonsai1_dequantize(const uint32_t* k_bits, const uint16_t* k_scale, const uint32_t* v_bits,
                                           const uint16_t* v_scale, int64_t n_rows, int head_dim, void* k_out,
                                           void* v_out, tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_bonsai1_dequantize");
  using namespace tq;
  if (n_rows < 0 || head_dim < kBonsaiGroup || head_dim % kBonsaiGroup)
    return set_error(TQ_ERR_INVALID_ARG, "bonsai1: n_rows >= 0 and head_dim a multiple of 128");
  if ((k_out && (!k_bits || !k_scale)) || (v_out && (!v_bits || !v_scale)))
    return set_error(TQ_ERR_INVALID_ARG, "bonsai1: NULL input");
  if (misaligned(k_out, 16) || misaligned(v_out, 16) || misaligned(k_bits, 4) || misaligned(v_bits, 4) ||
      misaligned(k_scale, 2) || misaligned(v_scale, 2))
    return set_error(TQ_ERR_INVALID_ARG, "bonsai1: outputs 16-byte and bits 4-byte aligned");
  BonsaiDeqArgs a{};
  a.bits[0] = k_out ? k_bits : nullptr;
  a.bits[1] = v_out ? v_bits : nullptr;
  a.scale[0] = k_scale;
  a.scale[1] = v_scale;
  a.out[0] = static_cast<uint4*>(k_out);
  a.out[1] = static_cast<uint4*>(v_out);
  a.n_words = n_rows * (head_dim / 32);
  if ((!k_out && !v_out) || a.n_words == 0) return set_error(TQ_OK, "");
  const long long blocks = blocks_for(2 * 4 * a.n_words);
  if (blocks > INT32_MAX) return set_error(TQ_ERR_INVALID_ARG, "bonsai1: too many rows for one launch");
  k_bonsai1_dequantize<<<(unsigned)blocks, kCodecThreads, 0, (cudaStream_t)stream>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(TQ_ERR_CUDA, cudaGetErrorString(e));
  return set_error(TQ_OK, "");
}
