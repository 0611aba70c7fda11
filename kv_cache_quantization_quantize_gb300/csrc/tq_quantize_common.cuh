// CUDA-core coder of the quantize-on-append pipeline ([Guide] §二, five steps), shared by the append
// kernels and by the decode-step kernel (which codes a ring block the moment it fills): source loads from
// the ring or the new input, the per-token coding of one 32-token block, and the packing of its page words.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cuda.h>

#include "tq_device.cuh"

namespace tq {

constexpr int kQThreads = 256;  // 8 warps; warp w quantises tokens w, w + 8, ...

struct AppendArgs {
  LayerView lv;
  const void* k;
  const void* v;
  int dt;  // 0 = bf16, 1 = f32
  const int32_t* seq_ids;
  const int32_t* n_new;  // per row; nullptr: one new token per row
  int max_new;
  int flush;  // 1: quantise the current ring block (tq_ring_flush)
  int full;   // 1: full_tq mode (ring_size 0): every appended token is quantised by the append itself
  // Wait-timeout test hook of the tcgen05 coders (tq_debug_append_wait_fault): the TMA copy of page task
  // fault_task ((row * Hkv + head) * pages per row + page of the append) is not issued, nor its expected
  // bytes, and the wait on it gives up after fault_polls polls. -1 in normal use.
  int fault_task = -1;
  uint32_t fault_polls = 0;
};

// Tensor map of k or v ([batch][max_new][Hkv][d] bf16) for the tcgen05 coders' page loads (tq_quantize.cu).
cudaError_t bulk_tensor_map(const void* base, int batch, int max_new, int hkv, int d, CUtensorMap* m);
// The head_dim 256 tcgen05 bulk coder (tq_quantize256.cu): `pages` page tasks per row, one persistent
// CTA per SM (`sms`).
cudaError_t launch_quantize_bulk256(const AppendArgs& a, int batch, int pages, int sms, cudaStream_t s);

namespace {

// New tokens of row b: n_new[b], or one per row when n_new is null (a decode step's append).
__device__ __forceinline__ int new_count(const AppendArgs& a, int b) { return a.n_new ? a.n_new[b] : 1; }

// Load 2 consecutive coordinates of one token of the source stream (ring bf16 or input bf16/f32).
__device__ __forceinline__ void load2(const AppendArgs& a, int which, int slot, int b, int h, int pos, int L, int Np,
                                      int j, float (&o)[2]) {
  const int d = a.lv.d;
  uint32_t u;
  if (pos < L) {  // still in the ring: ring index pos - Np
    u = *reinterpret_cast<const uint32_t*>(a.lv.ring + ((((size_t)slot * a.lv.Hkv + h) * 2 + which) * kPage + (pos - Np)) * d + j);
  } else {
    const size_t off = (((size_t)b * a.max_new + (pos - L)) * a.lv.Hkv + h) * d + j;
    const void* base = which ? a.v : a.k;
    if (a.dt != 0) {
      const float2 f = *reinterpret_cast<const float2*>(static_cast<const float*>(base) + off);
      o[0] = f.x;
      o[1] = f.y;
      return;
    }
    u = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(base) + off);
  }
  o[0] = __uint_as_float(u << 16);
  o[1] = __uint_as_float(u & 0xffff0000u);
}

// Load 4 consecutive coordinates of one token of the source stream (ring bf16 or input bf16/f32).
__device__ __forceinline__ void load4(const AppendArgs& a, int which, int slot, int b, int h, int pos, int L, int Np,
                                      int j, float (&o)[4]) {
  const int d = a.lv.d;
  if (pos < L) {  // still in the ring: ring index pos - Np
    const uint16_t* src = a.lv.ring + ((((size_t)slot * a.lv.Hkv + h) * 2 + which) * kPage + (pos - Np)) * d + j;
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    o[0] = __uint_as_float(u.x << 16);
    o[1] = __uint_as_float(u.x & 0xffff0000u);
    o[2] = __uint_as_float(u.y << 16);
    o[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    const size_t off = (((size_t)b * a.max_new + (pos - L)) * a.lv.Hkv + h) * d + j;
    const void* base = which ? a.v : a.k;
    if (a.dt == 0) {
      const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + off);
      o[0] = __uint_as_float(u.x << 16);
      o[1] = __uint_as_float(u.x & 0xffff0000u);
      o[2] = __uint_as_float(u.y << 16);
      o[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
      const float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
      o[0] = f.x;
      o[1] = f.y;
      o[2] = f.z;
      o[3] = f.w;
    }
  }
}

// Bits of plane pi of one token's key codes kc (coordinates 16 sq + 8 sub + 2c + e of a 128-coordinate
// half, sq < nsq) at bit 2 sq + sub + 16 e (+ shift) of a KBITS word (see kbit_loc).
__device__ __forceinline__ uint32_t kbits_field(const uint8_t* kc, int pi, int kb, int nsq, int shift) {
  uint32_t word = 0;
  for (int sq = 0; sq < nsq; ++sq)
#pragma unroll
    for (int sub = 0; sub < 2; ++sub)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        word |= (uint32_t)plane_bit(kc[16 * sq + 8 * sub + e], pi, kb) << (2 * sq + sub + 16 * e + shift);
      }
  return word;
}

// One token of the source stream in the lane_coord layout (D / 32 values per lane).
template <int D>
__device__ __forceinline__ void load_token(const AppendArgs& a, int which, int slot, int b, int h, int pos, int L,
                                           int Np, int lane, float (&x)[D / 32]) {
  if (D == 64) {
    float o[2];
    load2(a, which, slot, b, h, pos, L, Np, 2 * lane, o);
    x[0] = o[0];
    x[D / 32 - 1] = o[1];
  } else {
#pragma unroll
    for (int hh = 0; hh < D / 128; ++hh) {
      float o[4];
      load4(a, which, slot, b, h, pos, L, Np, 128 * hh + 4 * lane, o);
#pragma unroll
      for (int e = 0; e < 4; ++e) x[(4 * hh + e) % (D / 32)] = o[e];
    }
  }
}

// Shared-memory arrays of the CUDA-core quantiser for one 32-token block (a CTA codes one block at a
// time; row i is the block's token i): key codes (idx | sign << (kb - 1)), value codes, {n, gamma},
// value scales, and the f16 hi / lo split of the residuals (rows padded by 8 halves: conflict-free
// B-fragment reads).
template <int D>
constexpr int kRStride = D + 8;
template <int D>
struct QSmem {
  uint8_t* kcode;    // [32][D]
  uint8_t* vcode;    // [32][D]
  uint32_t* norms;   // [32] n16 | gamma16 << 16
  uint16_t* scales;  // [32][D/32]
  __half* rh;        // [32][kRStride] residual * 2^8, f16
  __half* rl;        // [32][kRStride] residual * 2^8 - rh, f16
  __device__ explicit QSmem(uint8_t* smem)
      : kcode(smem),
        vcode(kcode + 32 * D),
        norms(reinterpret_cast<uint32_t*>(vcode + 32 * D)),
        scales(reinterpret_cast<uint16_t*>(norms + 32)),
        rh(reinterpret_cast<__half*>(scales + 32 * (D / 32))),
        rl(rh + 32 * kRStride<D>) {}
};
template <int D>
constexpr size_t quantize_smem_bytes_d() {
  return 2 * 32 * D + 4 * 32 + 2 * 32 * (D / 32) + 2 * 2 * 32 * kRStride<D>;
}

// Mid-rise value code clamp(floor(fl(x / s)), -2^(vb-1), 2^(vb-1) - 1) + 2^(vb-1) for a scale s > 0 (the
// decision of an IEEE division rounded to nearest), without a division on the common path:
//   2 bits: three comparisons, code = [x >= -s] + [x >= 0] + [x >= s]. fl(x / s) >= -1 exactly when
//     x / s >= -(1 + 2^-24) (the midpoint below -1 rounds to the even -1), and no fp32 lies strictly between
//     -s (1 + 2^-24) and -s (the fp32 next to -s is an ulp of s > s 2^-24 away), so for fp32 x that is
//     x >= -s. Likewise fl(x / s) >= 1 exactly when x / s >= 1 - 2^-25, i.e. x >= s, and fl(x / s) >= 0
//     exactly when x >= 0.
//   4 bits: the floor of x * (1 / s), which lies within a few ulps of the rounded quotient, so it is
//     exact unless the product is within 4 ulps of an integer; those take the division.
__device__ __forceinline__ int value_code(float x, float s, float rcp, int vb) {
  if (vb == 2)
    return (int)(x >= -s) + (int)(x >= 0.f) + (int)(x >= s);
  const int vhalf = 1 << (vb - 1);
  const float qv = x * rcp;
  float fq = floorf(qv);
  const float fr = qv - fq, eps = fabsf(qv) * 4.8e-7f + 1e-30f;
  if (fr < eps || fr > 1.f - eps) fq = floorf(__fdiv_rn(x, s));
  return (int)fminf(fmaxf(fq, (float)-vhalf), (float)(vhalf - 1)) + vhalf;
}

// D += A B, m16n8k16, f16 operands, f32 accumulate.
__device__ __forceinline__ void mma_f16_acc(float (&c)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// Codes tokens [t_begin, t_end) of page pg of (row b, KV head h), all inside one 32-token block, into
// the shared-memory arrays: one warp per token for the norm, rotation, index, residual and value
// codes, then the QJL projection z = S r of the whole block as one f16 mma.sync GEMM (A = S from the
// f16 fragment table, B = the residuals scaled by 2^8 and split into f16 hi + lo; the scale leaves the
// signs unchanged). The page's first `valid` tokens come from the ring (positions below L) and then
// from the new input; tokens past `valid` are coded as zero vectors. Run by all NT threads of
// the CTA (a multiple of 32); ends with a block barrier. KB = key bits: a (KB - 1)-bit Lloyd-Max index plus the sign.
template <int D, int KB, int NT = kQThreads>
__device__ __forceinline__ void code_tokens(const AppendArgs& a, int b, int h, int slot, int L, int Np, int pg,
                                            int valid, int t_begin, int t_end, const QSmem<D>& sm) {
  constexpr int NE = D / 32;  // coordinates per lane
  constexpr int RS = kRStride<D>;
  uint8_t* kcode = sm.kcode;
  uint8_t* vcode = sm.vcode;
  uint32_t* norms = sm.norms;
  uint16_t* scales = sm.scales;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tb = t_begin & ~31;  // the block's first token
  const LayerView& lv = a.lv;
  constexpr int NL = 1 << (KB - 1);  // Lloyd-Max levels
  float Dv[NE], cent[NL], bnd[NL - 1];
#pragma unroll
  for (int e = 0; e < NE; ++e) Dv[e] = lv.D[lane_coord<D>(e, lane)];
#pragma unroll
  for (int i = 0; i < NL; ++i) cent[i] = lv.cb[kCbCent + i];
#pragma unroll
  for (int i = 0; i < NL - 1; ++i) bnd[i] = lv.cb[kCbBnd + i];

  const int vb = lv.vb, vhalf = 1 << (vb - 1);
  const float inv_sqrt_d = rsqrtf((float)D);
  for (int t = t_begin + warp; t < t_end; t += NT / 32) {
    const int pos = pg * kPage + t;
    float x[NE], y[NE];
    if (t < valid) {
      load_token<D>(a, 0, slot, b, h, pos, L, Np, lane, x);
    } else {
#pragma unroll
      for (int e = 0; e < NE; ++e) x[e] = 0.f;
    }
    // ---- key: n = ||k||, y = Pi k / n, Lloyd-Max index, residual, gamma ----
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < NE; ++e) ss = fmaf(x[e], x[e], ss);
    ss = warp_sum(ss);
    const float n = sqrtf(ss);
#pragma unroll
    for (int e = 0; e < NE; ++e) y[e] = x[e] * Dv[e];
    warp_fwht<NE>(y, lane);
    const float scale = n > 0.f ? 1.0f / (n * sqrtf((float)D)) : 0.f;
    float rr = 0.f;
    uint8_t* kc = kcode + (t - tb) * D;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const float yy = y[e] * scale;
      // index = #{boundaries below yy} by binary search over the sorted boundaries
      int idx;
      float cv;
      if (KB == 3) {
        const bool hb = yy > bnd[1];
        const bool lb = yy > (hb ? bnd[2] : bnd[0]);
        idx = 2 * hb + lb;
        cv = hb ? (lb ? cent[3] : cent[2]) : (lb ? cent[1] : cent[0]);
      } else {
        const bool b2 = yy > bnd[3];
        const bool b1 = yy > (b2 ? bnd[5] : bnd[1]);
        const bool b0 = yy > (b2 ? (b1 ? bnd[6] : bnd[4]) : (b1 ? bnd[2] : bnd[0]));
        idx = 4 * b2 + 2 * b1 + b0;
        cv = b2 ? (b1 ? (b0 ? cent[7] : cent[6]) : (b0 ? cent[5] : cent[4]))
                : (b1 ? (b0 ? cent[3] : cent[2]) : (b0 ? cent[1] : cent[0]));
      }
      const float res = yy - cv;
      rr = fmaf(res, res, rr);
      const int j = lane_coord<D>(e, lane);
      const float rs = res * 256.f;
      const __half hi = __float2half_rn(rs);
      sm.rh[(t - tb) * RS + j] = hi;
      sm.rl[(t - tb) * RS + j] = __float2half_rn(rs - __half2float(hi));
      kc[j] = (uint8_t)idx;
    }
    rr = warp_sum(rr);
    const float gamma = sqrtf(rr);
    if (lane == 0) {
      const __half nh = __float2half_rn(fminf(n, 65504.f)), gh = __float2half_rn(gamma);
      norms[t - tb] = (uint32_t)__half_as_ushort(nh) | ((uint32_t)__half_as_ushort(gh) << 16);
    }
    // ---- value: v' = Pi v, symmetric mid-rise groups of 32, fp16 scale ----
    if (t < valid) {
      load_token<D>(a, 1, slot, b, h, pos, L, Np, lane, x);
#pragma unroll
      for (int e = 0; e < NE; ++e) x[e] *= Dv[e];
    } else {
#pragma unroll
      for (int e = 0; e < NE; ++e) x[e] = 0.f;
    }
    warp_fwht<NE>(x, lane);
    uint8_t* vc = vcode + (t - tb) * D;
    if (D == 64) {  // a group of 32 coordinates is 16 lanes x 2
      float am = 0.f;
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        x[e] *= inv_sqrt_d;
        am = fmaxf(am, fabsf(x[e]));
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      const float s32 = fminf(__fdiv_rn(am, (float)vhalf - 0.5f), 65504.f);
      const __half sh = __float2half_rn(s32);
      const float s = __half2float(sh), rcp = s > 0.f ? __frcp_rn(s) : 0.f;
#pragma unroll
      for (int e = 0; e < NE; ++e)
        vc[lane_coord<D>(e, lane)] = (uint8_t)(s > 0.f ? value_code(x[e], s, rcp, vb) : vhalf);
      if ((lane & 15) == 0) scales[(t - tb) * (D / 32) + (lane >> 4)] = __half_as_ushort(sh);
    }
#pragma unroll
    for (int hh = 0; hh < (D == 64 ? 0 : NE / 4); ++hh) {
      float am = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[4 * hh + e] *= inv_sqrt_d;
        am = fmaxf(am, fabsf(x[4 * hh + e]));
      }
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
      const float s32 = fminf(__fdiv_rn(am, (float)vhalf - 0.5f), 65504.f);
      const __half sh = __float2half_rn(s32);
      const float s = __half2float(sh), rcp = s > 0.f ? __frcp_rn(s) : 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        vc[128 * hh + 4 * lane + e] = (uint8_t)(s > 0.f ? value_code(x[4 * hh + e], s, rcp, vb) : vhalf);
      if ((lane & 7) == 0) scales[(t - tb) * (D / 32) + 4 * hh + (lane >> 3)] = __half_as_ushort(sh);
    }
  }
  __syncthreads();
  // ---- QJL: Z^T = S R^T for the block; warp task = one 16-row m-tile of S x NTW 8-token n-tiles ----
  {
    constexpr int MTS = D / 16, NTW = D >= 128 ? 4 : 2;
    const int g = lane >> 2, c = lane & 3;
    for (int u = warp; u < MTS * (4 / NTW); u += NT / 32) {
      const int mt = u % MTS, nt0 = (u / MTS) * NTW;
      float z[NTW][4];
#pragma unroll
      for (int n = 0; n < NTW; ++n) z[n][0] = z[n][1] = z[n][2] = z[n][3] = 0.f;
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint4 A = lv.S_frag[sfrag_idx(D, mt, ks, lane)];
#pragma unroll
        for (int n = 0; n < NTW; ++n) {
          const int row = (8 * (nt0 + n) + g) * RS + 16 * ks + 2 * c;
          mma_f16_acc(z[n], A, *reinterpret_cast<const uint32_t*>(sm.rh + row),
                      *reinterpret_cast<const uint32_t*>(sm.rh + row + 8));
          mma_f16_acc(z[n], A, *reinterpret_cast<const uint32_t*>(sm.rl + row),
                      *reinterpret_cast<const uint32_t*>(sm.rl + row + 8));
        }
      }
#pragma unroll
      for (int n = 0; n < NTW; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = tb + 8 * (nt0 + n) + 2 * c + (i & 1), row = 16 * mt + g + 8 * (i >> 1);
          if (t >= t_begin && t < t_end)
            kcode[(t - tb) * D + row] = (uint8_t)(kcode[(t - tb) * D + row] | ((z[n][i] >= 0.f) << (KB - 1)));
        }
    }
  }
  __syncthreads();
}

// Quantises the 32-token block q32 of page pg of (row b, KV head h): the page's first `valid` tokens
// come from the ring (positions below L) and then from the new input; tokens past `valid` are coded as
// zero vectors. A 32-token block owns whole words of every page section, so four CTAs can write the
// four blocks of one page independently. Run by all NT threads of the CTA.
template <int D, int KB, int NT = kQThreads>
__device__ __forceinline__ void quantize_page_cta(const AppendArgs& a, int b, int h, int slot, int L, int Np, int pg,
                                                  int valid, int q32, uint8_t* smem) {
  const int t0 = 32 * q32, t1 = t0 + 32;
  const QSmem<D> sm(smem);
  code_tokens<D, KB, NT>(a, b, h, slot, L, Np, pg, valid, t0, t1, sm);
  uint8_t* kcode = sm.kcode;
  uint8_t* vcode = sm.vcode;
  uint32_t* norms = sm.norms;
  uint16_t* scales = sm.scales;
  const int tid = threadIdx.x;
  const LayerView& lv = a.lv;
  const int vb = lv.vb;

  // ---- pack the page (fragment-major layout) ----
  uint8_t* page = page_addr(lv, slot, h, pg);
  if (!page) {  // paged cache without a block for this page: nothing is written
    if (tid == 0) set_status(lv.status, TQ_DEV_ERR_BLOCK);
    return;
  }
  const PageLayout pl = page_layout(D, vb, KB);
  uint32_t* kw = reinterpret_cast<uint32_t*>(page + pl.kbits_off);
  constexpr int HALVES = D >= 128 ? D / 128 : 1;  // 128-coordinate halves (the head_dim 64 words are below)
  constexpr int WT = 64 * KB;                      // KBITS words of a tile per half (a 32-token group at d=64)
  if (D == 64) {  // one word holds both 16-token tiles of the block: [group][plane][lane][row]
    for (int w = q32 * WT + tid; w < (q32 + 1) * WT; w += NT) {
      const int r = w & 1, ln = (w >> 1) & 31, pi = (w >> 6) % KB;
      uint32_t word = 0;
#pragma unroll
      for (int kap = 0; kap < 2; ++kap)
        word |= kbits_field(kcode + (16 * kap + (ln >> 2) + 8 * r) * D + 2 * (ln & 3), pi, KB, 4, 8 * kap);
      kw[w] = word;
    }
  }
  for (int w = (t0 / 16) * WT * HALVES + tid; D >= 128 && w < (t1 / 16) * WT * HALVES; w += NT) {
    const int r = w & 1, ln = (w >> 1) & 31, hf = (w >> 6) % HALVES, pi = (w / (64 * HALVES)) % KB;
    const int tile = w / (WT * HALVES);
    const int t = 16 * tile + (ln >> 2) + 8 * r, c = ln & 3;
    kw[w] = kbits_field(kcode + (t - t0) * D + 128 * hf + 2 * c, pi, KB, 8, 0);
  }
  uint32_t* nw = reinterpret_cast<uint32_t*>(page + pl.norms_off);
  for (int t = t0 + tid; t < t1; t += NT) nw[t] = norms[t - t0];
  uint32_t* vw = reinterpret_cast<uint32_t*>(page + pl.vbits_off);
  if (vb == 2) {
    for (int w = q32 * (D / 16) * 32 + tid; w < (q32 + 1) * (D / 16) * 32; w += NT) {
      const int ln = w & 31, mt = (w >> 5) % (D / 16), blk = w / (32 * (D / 16));
      const int g = ln >> 2, c = ln & 3;
      uint32_t word = 0;
#pragma unroll
      for (int kap = 0; kap < 2; ++kap)
#pragma unroll
        for (int rg = 0; rg < 4; ++rg)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int t = 32 * blk + 16 * kap + 8 * (rg >> 1) + 2 * c + e;
            const int j = 16 * mt + 8 * (rg & 1) + g;
            word |= (uint32_t)vcode[(t - t0) * D + j] << (16 * e + 2 * vfield2(kap, rg));
          }
      vw[w] = word;
    }
  } else {
    for (int w = q32 * (D / 16) * 64 + tid; w < (q32 + 1) * (D / 16) * 64; w += NT) {
      const int kap = w & 1, ln = (w >> 1) & 31, mt = (w >> 6) % (D / 16), blk = w / (64 * (D / 16));
      const int g = ln >> 2, c = ln & 3;
      uint32_t word = 0;
#pragma unroll
      for (int rg = 0; rg < 4; ++rg)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 32 * blk + 16 * kap + 8 * (rg >> 1) + 2 * c + e;
          const int j = 16 * mt + 8 * (rg & 1) + g;
          word |= (uint32_t)vcode[(t - t0) * D + j] << (16 * e + 4 * vfield4(rg));
        }
      vw[w] = word;
    }
  }
  uint16_t* sw = reinterpret_cast<uint16_t*>(page + pl.vscale_off);
  for (int i = t0 * (D / 32) + tid; i < t1 * (D / 32); i += NT)
    sw[vscale_idx(D, i / (D / 32), i % (D / 32))] = scales[i - t0 * (D / 32)];
}

// Which page this CTA writes, from the sequence state. Returns false when the CTA has no work.
// An append codes every 128-token block that it completes, including the one that fills the ring to
// 128 tokens (those stay in the ring as well until the next token starts a new ring block). So the
// blocks below 128 floor(L / 128) are always coded, and a ring that rolls over finds its block coded.
__device__ __forceinline__ bool page_task(const AppendArgs& a, int b, int j, int& slot, int& L, int& Np, int& pg,
                                          int& valid, bool report) {
  slot = a.seq_ids[b];
  if (slot < 0 || slot >= a.lv.max_seqs) {
    if (report) set_status(a.lv.status, TQ_DEV_ERR_SEQ_ID);
    return false;
  }
  L = a.lv.state[2 * slot];
  Np = L > 0 ? kPage * ((L - 1) / kPage) : 0;
  if (a.flush) {
    const int R = L - Np;
    if (R <= 0 || j > 0) return false;
    pg = Np / kPage;
    valid = R;
    return true;
  }
  const int nn = new_count(a, b);
  const int L2 = L + nn;
  if (nn < 0 || nn > a.max_new || L2 > a.lv.max_ctx) {
    if (report) set_status(a.lv.status, TQ_DEV_ERR_CAPACITY);
    return false;
  }
  const int C = kPage * (L / kPage), C2 = kPage * (L2 / kPage);  // complete blocks before and after
  if (j >= (C2 - C) / kPage) return false;
  pg = C / kPage + j;
  valid = kPage;
  return true;
}

// After the page loop of a persistent tcgen05 coder (thread 0): every copy or MMA batch armed on one
// of the CTA's barriers and not seen complete by the thread that counts it is waited for (bounded), so
// that nothing lands in shared memory or TMEM after the CTA frees them. armed / done: per barrier, the
// phases armed and the phases seen complete. In a run without a failed wait the counts are equal.
// Slot `skip` of the n barrier slots holds the TMEM address. Returns false if a wait gives up here too.
__device__ __forceinline__ bool bulk_drain(uint64_t* bars, int n, int skip, uint32_t* armed, uint32_t* done) {
  bool ok = true;
  for (int i = 0; i < n; ++i) {
    if (i == skip) continue;  // the TMEM address slot
    while (done[i] < armed[i]) {
      if (!mbar_wait(bars + i, done[i] & 1u)) {
        ok = false;
        break;
      }
      ++done[i];
    }
  }
  return ok;
}

// The pages one row of a bulk append writes (page_task's per-row part, for appends): its slot, L and the
// page count (from page L / 128 on); npages = 0 for a row with a bad sequence id or capacity (reported
// when `report`). b = -1: nothing cached yet.
struct RowTask {
  int b = -1, slot = 0, L = 0, npages = 0;
};
__device__ __forceinline__ void row_task(const AppendArgs& a, int b, RowTask& r, bool report) {
  r.b = b;
  r.npages = 0;
  r.slot = a.seq_ids[b];
  if (r.slot < 0 || r.slot >= a.lv.max_seqs) {
    if (report) set_status(a.lv.status, TQ_DEV_ERR_SEQ_ID);
    return;
  }
  r.L = a.lv.state[2 * r.slot];
  const int nn = new_count(a, b), L2 = r.L + nn;
  if (nn < 0 || nn > a.max_new || L2 > a.lv.max_ctx) {
    if (report) set_status(a.lv.status, TQ_DEV_ERR_CAPACITY);
    return;
  }
  r.npages = L2 / kPage - r.L / kPage;  // complete blocks after the append minus those before (as page_task)
}

// Next task (>= task, stepping by the grid) that has a page to write, or ntasks; for appends (not
// flushes). The row lookup is cached in rc, so a CTA whose tasks stay in one row reads the row's state
// once. Thread `reporter` of the CTA reports a row's bad sequence id or capacity (at the row's first
// task, which is also the first task of that row any CTA visits).
__device__ __forceinline__ int bulk_next(const AppendArgs& a, int task, int ntasks, int pages_per_row, RowTask& rc,
                                         int& b, int& h, int& slot, int& L, int& Np, int& pg, int reporter = 0) {
  for (; task < ntasks; task += gridDim.x) {
    b = task / (a.lv.Hkv * pages_per_row);
    h = (task / pages_per_row) % a.lv.Hkv;
    const int j = task % pages_per_row;
    if (b != rc.b) row_task(a, b, rc, h == 0 && j == 0 && (int)threadIdx.x == reporter);
    if (j >= rc.npages) continue;
    slot = rc.slot;
    L = rc.L;
    Np = L > 0 ? kPage * ((L - 1) / kPage) : 0;
    pg = L / kPage + j;
    return task;
  }
  return ntasks;
}

}  // namespace
}  // namespace tq
