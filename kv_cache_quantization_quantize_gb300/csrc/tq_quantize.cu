// Quantize-on-append ([Guide] §二, five-step pipeline): one CTA writes one packed page (128 tokens of
// one KV head). This is the CUDA-core path for ring flushes and appends. The QJL projection z = S r
// is an fp32 FMA contraction against S^T staged in shared memory.
#include <algorithm>

#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kQThreads = 256;  // 8 warps; warp w quantises tokens w, w + 8, ...

struct AppendArgs {
  LayerView lv;
  const void* k;
  const void* v;
  int dt;  // 0 = bf16, 1 = f32
  const int32_t* seq_ids;
  const int32_t* n_new;
  int max_new;
  int flush;  // 1: quantise the current ring block (tq_ring_flush)
};

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

// Which page this CTA writes, from the sequence state. Returns false when the CTA has no work.
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
  const int nn = a.n_new[b];
  const int L2 = L + nn;
  if (nn < 0 || nn > a.max_new || L2 > a.lv.max_ctx) {
    if (report) set_status(a.lv.status, TQ_DEV_ERR_CAPACITY);
    return false;
  }
  const int Np2 = L2 > 0 ? kPage * ((L2 - 1) / kPage) : 0;
  if (j >= (Np2 - Np) / kPage) return false;
  pg = Np / kPage + j;
  valid = kPage;
  return true;
}

// Quantises page pg of (row b, KV head h): its first `valid` tokens come from the ring (positions
// below L) and then from the new input. Run by all kQThreads threads of the CTA.
template <int D>
__device__ __forceinline__ void quantize_page_cta(const AppendArgs& a, int b, int h, int slot, int L, int Np, int pg,
                                                  int valid, uint8_t* smem) {
  constexpr int NE = D / 32;  // coordinates per lane
  uint32_t* st2 = reinterpret_cast<uint32_t*>(smem);                    // S^T as bf16 pairs [D][D/2]
  uint8_t* kcode = smem + 2 * D * D;                                    // [128][D]: idx | sign << 2
  uint8_t* vcode = kcode + kPage * D;                                   // [128][D]
  uint32_t* norms = reinterpret_cast<uint32_t*>(vcode + kPage * D);     // [128] n16 | gamma16 << 16
  uint16_t* scales = reinterpret_cast<uint16_t*>(norms + kPage);        // [128][D/32]
  float* rbuf = reinterpret_cast<float*>(scales + kPage * (D / 32));    // [8 warps][D]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const LayerView& lv = a.lv;
  // stage S^T (bf16) in shared memory
  {
    const uint4* src = reinterpret_cast<const uint4*>(lv.St);
    uint4* dst = reinterpret_cast<uint4*>(st2);
    for (int i = tid; i < D * D / 8; i += kQThreads) dst[i] = src[i];
  }
  float Dv[NE], cent[4], bnd[3];
#pragma unroll
  for (int e = 0; e < NE; ++e) Dv[e] = lv.D[(e >> 2) * 128 + 4 * lane + (e & 3)];
#pragma unroll
  for (int i = 0; i < 4; ++i) cent[i] = lv.cb[i];
#pragma unroll
  for (int i = 0; i < 3; ++i) bnd[i] = lv.cb[4 + i];
  __syncthreads();

  const int vb = lv.vb, vhalf = 1 << (vb - 1);
  const float inv_sqrt_d = rsqrtf((float)D);
  float* r = rbuf + warp * D;
  for (int t = warp; t < kPage; t += kQThreads / 32) {
    const int pos = pg * kPage + t;
    float x[NE], y[NE];
    if (t < valid) {
#pragma unroll
      for (int hh = 0; hh < NE / 4; ++hh) {
        float o[4];
        load4(a, 0, slot, b, h, pos, L, Np, 128 * hh + 4 * lane, o);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[4 * hh + e] = o[e];
      }
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
    uint8_t* kc = kcode + t * D;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const float yy = y[e] * scale;
      const int idx = (yy > bnd[0]) + (yy > bnd[1]) + (yy > bnd[2]);
      const float res = yy - cent[idx];
      rr = fmaf(res, res, rr);
      const int j = (e >> 2) * 128 + 4 * lane + (e & 3);
      r[j] = res;
      kc[j] = (uint8_t)idx;
    }
    rr = warp_sum(rr);
    const float gamma = sqrtf(rr);
    __syncwarp();
    // ---- QJL: z = S r; lane owns rows 2l, 2l+1 (+64m) ----
    {
      constexpr int NR = D / 64;  // row pairs per lane
      float z0[NR], z1[NR];
#pragma unroll
      for (int m = 0; m < NR; ++m) z0[m] = z1[m] = 0.f;
      for (int jj = 0; jj < D; ++jj) {
        const float rj = r[jj];
#pragma unroll
        for (int m = 0; m < NR; ++m) {
          const uint32_t s = st2[jj * (D / 2) + lane + 32 * m];
          z0[m] = fmaf(__uint_as_float(s << 16), rj, z0[m]);
          z1[m] = fmaf(__uint_as_float(s & 0xffff0000u), rj, z1[m]);
        }
      }
      __syncwarp();
#pragma unroll
      for (int m = 0; m < NR; ++m) {
        const int i0 = 2 * lane + 64 * m;
        kc[i0] = (uint8_t)(kc[i0] | ((z0[m] >= 0.f) << 2));
        kc[i0 + 1] = (uint8_t)(kc[i0 + 1] | ((z1[m] >= 0.f) << 2));
      }
    }
    if (lane == 0) {
      const __half nh = __float2half_rn(fminf(n, 65504.f)), gh = __float2half_rn(gamma);
      norms[t] = (uint32_t)__half_as_ushort(nh) | ((uint32_t)__half_as_ushort(gh) << 16);
    }
    // ---- value: v' = Pi v, symmetric mid-rise groups of 32, fp16 scale ----
    if (t < valid) {
#pragma unroll
      for (int hh = 0; hh < NE / 4; ++hh) {
        float o[4];
        load4(a, 1, slot, b, h, pos, L, Np, 128 * hh + 4 * lane, o);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[4 * hh + e] = o[e] * Dv[4 * hh + e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < NE; ++e) x[e] = 0.f;
    }
    warp_fwht<NE>(x, lane);
    uint8_t* vc = vcode + t * D;
#pragma unroll
    for (int hh = 0; hh < NE / 4; ++hh) {
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
      const float s = __half2float(sh);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int code = vhalf;
        if (s > 0.f) {
          const float qv = floorf(__fdiv_rn(x[4 * hh + e], s));
          code = (int)fminf(fmaxf(qv, (float)-vhalf), (float)(vhalf - 1)) + vhalf;
        }
        vc[128 * hh + 4 * lane + e] = (uint8_t)code;
      }
      if ((lane & 7) == 0) scales[t * (D / 32) + 4 * hh + (lane >> 3)] = __half_as_ushort(sh);
    }
  }
  __syncthreads();

  // ---- pack the page (fragment-major layout) ----
  uint8_t* page = lv.pages + (((size_t)slot * lv.Hkv + h) * lv.max_pages + pg) * lv.page_bytes;
  const PageLayout pl = page_layout(D, vb);
  uint32_t* kw = reinterpret_cast<uint32_t*>(page + pl.kbits_off);
  constexpr int HALVES = D / 128;
  for (int w = tid; w < 8 * 3 * HALVES * 32 * 2; w += kQThreads) {
    const int r = w & 1, ln = (w >> 1) & 31, hf = (w >> 6) % HALVES, pi = (w / (64 * HALVES)) % 3;
    const int tile = w / (192 * HALVES);
    const int t = 16 * tile + (ln >> 2) + 8 * r, c = ln & 3;
    const uint8_t* kc = kcode + t * D + 128 * hf + 2 * c;
    uint32_t word = 0;
#pragma unroll
    for (int sq = 0; sq < 8; ++sq)
#pragma unroll
      for (int sub = 0; sub < 2; ++sub)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int code = kc[16 * sq + 8 * sub + e];
          const int bit = pi == 0 ? (code >> 1) & 1 : pi == 1 ? code & 1 : (code >> 2) & 1;
          word |= (uint32_t)bit << (2 * sq + sub + 16 * e);
        }
    kw[w] = word;
  }
  uint32_t* nw = reinterpret_cast<uint32_t*>(page + pl.norms_off);
  for (int t = tid; t < kPage; t += kQThreads) nw[t] = norms[t];
  uint32_t* vw = reinterpret_cast<uint32_t*>(page + pl.vbits_off);
  if (vb == 2) {
    for (int w = tid; w < 4 * (D / 16) * 32; w += kQThreads) {
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
            word |= (uint32_t)vcode[t * D + j] << (16 * e + 2 * vfield2(kap, rg));
          }
      vw[w] = word;
    }
  } else {
    for (int w = tid; w < 4 * (D / 16) * 32 * 2; w += kQThreads) {
      const int kap = w & 1, ln = (w >> 1) & 31, mt = (w >> 6) % (D / 16), blk = w / (64 * (D / 16));
      const int g = ln >> 2, c = ln & 3;
      uint32_t word = 0;
#pragma unroll
      for (int rg = 0; rg < 4; ++rg)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 32 * blk + 16 * kap + 8 * (rg >> 1) + 2 * c + e;
          const int j = 16 * mt + 8 * (rg & 1) + g;
          word |= (uint32_t)vcode[t * D + j] << (16 * e + 4 * vfield4(rg));
        }
      vw[w] = word;
    }
  }
  uint16_t* sw = reinterpret_cast<uint16_t*>(page + pl.vscale_off);
  for (int i = tid; i < kPage * (D / 32); i += kQThreads) sw[vscale_idx(D, i / (D / 32), i % (D / 32))] = scales[i];
}

template <int D>
__global__ void __launch_bounds__(kQThreads) k_quantize_pages(AppendArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int b = blockIdx.x, h = blockIdx.y;
  pdl_wait();  // sequence state, ring and inputs come from earlier work on the stream
  pdl_launch();
  int slot, L, Np, pg, valid;
  if (!page_task(a, b, blockIdx.z, slot, L, Np, pg, valid, h == 0 && blockIdx.z == 0 && threadIdx.x == 0)) return;
  quantize_page_cta<D>(a, b, h, slot, L, Np, pg, valid, smem);
}

// Appends of fewer than 128 tokens per row in one launch: CTA (row b, KV head h) packs the page that
// completes when the ring overflows (at most one), then writes head h's new ring rows. The last CTA
// of the row to arrive publishes the new length. Dependents (the decode) are released only after
// that, so they may read the state before their own stream wait.
template <int D>
__global__ void __launch_bounds__(kQThreads) k_append_small(AppendArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  pdl_wait();  // sequence state, ring and inputs come from earlier work on the stream
  const LayerView& lv = a.lv;
  const int slot = a.seq_ids[b];
  if (slot < 0 || slot >= lv.max_seqs) {
    if (h == 0 && tid == 0) set_status(lv.status, TQ_DEV_ERR_SEQ_ID);
    return;
  }
  const int L = lv.state[2 * slot], F = lv.state[2 * slot + 1];
  const int Np = L > 0 ? kPage * ((L - 1) / kPage) : 0;
  const int nn = a.n_new[b];
  const int L2 = L + nn;
  if (nn < 0 || nn > a.max_new || L2 > lv.max_ctx) {
    if (h == 0 && tid == 0) set_status(lv.status, TQ_DEV_ERR_CAPACITY);
    return;
  }
  const int Np2 = L2 > 0 ? kPage * ((L2 - 1) / kPage) : 0;
  if (Np2 > Np) quantize_page_cta<D>(a, b, h, slot, L, Np, Np / kPage, kPage, smem);  // Np2 - Np == 128
  __syncthreads();  // the page read the old ring rows of head h
  const int p0 = max(L, Np2);
  const int d = lv.d, q4 = d / 4;
  const int n_items = (L2 - p0) * 2 * q4;  // (pos, which, quad) of head h
  for (int it = tid; it < n_items; it += blockDim.x) {
    const int quad = it % q4, which = (it / q4) & 1, pos = p0 + it / (2 * q4);
    const size_t src = (((size_t)b * a.max_new + (pos - L)) * lv.Hkv + h) * d + 4 * quad;
    uint16_t* dst = lv.ring + ((((size_t)slot * lv.Hkv + h) * 2 + which) * kPage + (pos - Np2)) * d + 4 * quad;
    const void* base = which ? a.v : a.k;
    uint2 out;
    if (a.dt == 0) {
      out = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + src);
    } else {
      const float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + src);
      out.x = (uint32_t)f32_to_bf16_rn(f.x) | ((uint32_t)f32_to_bf16_rn(f.y) << 16);
      out.y = (uint32_t)f32_to_bf16_rn(f.z) | ((uint32_t)f32_to_bf16_rn(f.w) << 16);
    }
    *reinterpret_cast<uint2*>(dst) = out;
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(lv.acnt + slot, 1);
    if (old == lv.Hkv - 1) {  // every head of the row is done with the old state
      lv.acnt[slot] = 0;
      lv.state[2 * slot] = L2;
      lv.state[2 * slot + 1] = Np2 > Np ? 0 : F;
      __threadfence();
    }
  }
  __syncthreads();
  pdl_launch();
}

// =============================================================================================
// Bulk quantise (head_dim 128): the QJL projection z = S r on tcgen05 tensor cores.
//   - The residual r of a 128-token page is split into bf16 hi + lo (|r - hi - lo| <= 2^-18 |r|) and
//     written as operand A (128 tokens x 128 coordinates, K-major, 128-byte swizzle).
//   - S (operand B) is loaded once per persistent CTA from its pre-swizzled table.
//   - 16 MMAs (M = N = 128, K = 16; hi then lo) accumulate z in TMEM (fp32, 128 columns).
//   - Each thread reads back one token row with tcgen05.ld and keeps the signs.
// =============================================================================================
constexpr int kTcThreads = 256;
constexpr uint32_t kTcS = 0, kTcAhi = 32768, kTcAlo = 65536, kTcKcode = 98304, kTcVcode = kTcKcode + 16384;
constexpr uint32_t kTcSign = kTcVcode + 16384, kTcNorm = kTcSign + 2048, kTcScale = kTcNorm + 512;
constexpr uint32_t kTcBar = kTcScale + 1024, kTcEnd = kTcBar + 64;
constexpr size_t kTcSmem = kTcEnd + 1024;  // + alignment slack for the 1024-byte swizzle atoms

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  return (uint64_t)((smem_addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: D = f32, A = B = bf16, both K-major, N = 128, M = 128.
constexpr uint32_t kIdescBf16M128N128 = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes 32(w%4)..+31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1) k_quantize_bulk128(AppendArgs a, int pages_per_row, int batch) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* kcode = sm + kTcKcode;
  uint8_t* vcode = sm + kTcVcode;
  uint32_t* sgn = reinterpret_cast<uint32_t*>(sm + kTcSign);   // [128 tokens][4] sign words
  uint32_t* norms = reinterpret_cast<uint32_t*>(sm + kTcNorm);
  uint16_t* scales = reinterpret_cast<uint16_t*>(sm + kTcScale);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(sm + kTcBar);
  uint64_t* bar_mma = bar_s + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_s + 2);
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_launch();
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_mma, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    mbar_expect_tx(bar_s, 2u * D * D);
    bulk_g2s(sm + kTcS, lv.S_sw, 2u * D * D, bar_s);
  }
  if (warp == 0) {  // 128 TMEM columns: the fp32 accumulator of one 128 x 128 page
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;\n" ::"r"(smem_u32(tslot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  float Dv[4], cent[4], bnd[3];
#pragma unroll
  for (int e = 0; e < 4; ++e) Dv[e] = lv.D[4 * lane + e];
#pragma unroll
  for (int i = 0; i < 4; ++i) cent[i] = lv.cb[i];
#pragma unroll
  for (int i = 0; i < 3; ++i) bnd[i] = lv.cb[4 + i];
  bool ok = __syncthreads_and(mbar_wait(bar_s, 0)) != 0;
  const int vb = lv.vb, vhalf = 1 << (vb - 1);
  const float inv_sqrt_d = rsqrtf((float)D);
  const uint32_t s_addr = smem_u32(sm + kTcS), ahi_addr = smem_u32(sm + kTcAhi), alo_addr = smem_u32(sm + kTcAlo);
  uint32_t mma_phase = 0;
  const int ntasks = batch * lv.Hkv * pages_per_row;
  for (int task = blockIdx.x; ok && task < ntasks; task += gridDim.x) {
    const int b = task / (lv.Hkv * pages_per_row), h = (task / pages_per_row) % lv.Hkv, j = task % pages_per_row;
    int slot, L, Np, pg, valid;
    if (!page_task(a, b, j, slot, L, Np, pg, valid, h == 0 && j == 0 && tid == 0)) continue;  // CTA-uniform
    // ---- per token (warp): key rotation, norm, Lloyd-Max code, residual -> A; value quantisation.
    // The 16 tokens of a warp are handled in chunks of 8 whose K and V rows are loaded together. ----
    for (int c0 = 0; c0 < kPage / (kTcThreads / 32); c0 += 8) {
    float kx[8][4], vx[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = warp + (kTcThreads / 32) * (c0 + i);
      if (t < valid) {
        load4(a, 0, slot, b, h, pg * kPage + t, L, Np, 4 * lane, kx[i]);
        load4(a, 1, slot, b, h, pg * kPage + t, L, Np, 4 * lane, vx[i]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) kx[i][e] = vx[i][e] = 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = warp + (kTcThreads / 32) * (c0 + i);
      float x[4], y[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = kx[i][e];
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) ss = fmaf(x[e], x[e], ss);
      ss = warp_sum(ss);
      const float n = sqrtf(ss);
#pragma unroll
      for (int e = 0; e < 4; ++e) y[e] = x[e] * Dv[e];
      warp_fwht<4>(y, lane);
      const float scale = n > 0.f ? 1.0f / (n * sqrtf((float)D)) : 0.f;
      float rr = 0.f, res[4];
      uint32_t codes4 = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float yy = y[e] * scale;
        const int idx = (yy > bnd[0]) + (yy > bnd[1]) + (yy > bnd[2]);
        res[e] = yy - cent[idx];
        rr = fmaf(res[e], res[e], rr);
        codes4 |= (uint32_t)idx << (8 * e);
      }
      *reinterpret_cast<uint32_t*>(kcode + t * D + 4 * lane) = codes4;
      rr = warp_sum(rr);
      uint32_t hi[2], lo[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint16_t h0 = f32_to_bf16_rn(res[2 * e]), h1 = f32_to_bf16_rn(res[2 * e + 1]);
        const uint16_t l0 = f32_to_bf16_rn(res[2 * e] - bf16_to_f32(h0));
        const uint16_t l1 = f32_to_bf16_rn(res[2 * e + 1] - bf16_to_f32(h1));
        hi[e] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        lo[e] = (uint32_t)l0 | ((uint32_t)l1 << 16);
      }
      const uint32_t off = sw128_offset(t, 4 * lane);
      *reinterpret_cast<uint2*>(sm + kTcAhi + off) = make_uint2(hi[0], hi[1]);
      *reinterpret_cast<uint2*>(sm + kTcAlo + off) = make_uint2(lo[0], lo[1]);
      if (lane == 0) {
        const __half nh = __float2half_rn(fminf(n, 65504.f)), gh = __float2half_rn(sqrtf(rr));
        norms[t] = (uint32_t)__half_as_ushort(nh) | ((uint32_t)__half_as_ushort(gh) << 16);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = vx[i][e] * Dv[e];
      warp_fwht<4>(x, lane);
      float am = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[e] *= inv_sqrt_d;
        am = fmaxf(am, fabsf(x[e]));
      }
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
      const float s32 = fminf(__fdiv_rn(am, (float)vhalf - 0.5f), 65504.f);
      const __half sh = __float2half_rn(s32);
      const float sv = __half2float(sh);
      uint32_t vc4 = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int code = vhalf;
        if (sv > 0.f) {
          const float qv = floorf(__fdiv_rn(x[e], sv));
          code = (int)fminf(fmaxf(qv, (float)-vhalf), (float)(vhalf - 1)) + vhalf;
        }
        vc4 |= (uint32_t)code << (8 * e);
      }
      *reinterpret_cast<uint32_t*>(vcode + t * D + 4 * lane) = vc4;
      if ((lane & 7) == 0) scales[t * (D / 32) + (lane >> 3)] = __half_as_ushort(sh);
    }
    }
    // ---- z = S r on the tensor cores ----
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (ks >> 2) * 16384 + (ks & 3) * 32;
        umma_bf16(tmem, umma_desc_sw128(ahi_addr + koff), umma_desc_sw128(s_addr + koff), kIdescBf16M128N128,
                  ks > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (ks >> 2) * 16384 + (ks & 3) * 32;
        umma_bf16(tmem, umma_desc_sw128(alo_addr + koff), umma_desc_sw128(s_addr + koff), kIdescBf16M128N128, 1u);
      }
      umma_commit(bar_mma);
    }
    ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase)) != 0;
    mma_phase ^= 1;
    if (!ok) break;
    tc_fence_after();
    {  // warp w: TMEM lanes 32(w%4).. (tokens), columns 64(w/4).. (projection rows)
      const int q = warp & 3, ch = warp >> 2, t = 32 * q + lane;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t z[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(64 * ch + 32 * cc), z);
        uint32_t bits = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) bits |= (uint32_t)(__uint_as_float(z[i]) >= 0.f) << i;
        sgn[t * 4 + 2 * ch + cc] = bits;
      }
    }
    tc_fence_before();
    __syncthreads();
    // ---- pack the page (fragment-major layout) ----
    uint8_t* page = lv.pages + (((size_t)slot * lv.Hkv + h) * lv.max_pages + pg) * lv.page_bytes;
    const PageLayout pl = page_layout(D, vb);
    uint32_t* kw = reinterpret_cast<uint32_t*>(page + pl.kbits_off);
    for (int w = tid; w < 8 * 3 * 32 * 2; w += kTcThreads) {
      const int r = w & 1, ln = (w >> 1) & 31, pi = (w >> 6) % 3, tile = w / 192;
      const int t = 16 * tile + (ln >> 2) + 8 * r, c = ln & 3;
      uint32_t word = 0;
      if (pi < 2) {
        const uint8_t* kc = kcode + t * D + 2 * c;
#pragma unroll
        for (int sq = 0; sq < 8; ++sq)
#pragma unroll
          for (int sub = 0; sub < 2; ++sub)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int code = kc[16 * sq + 8 * sub + e];
              word |= (uint32_t)((pi == 0 ? code >> 1 : code) & 1) << (2 * sq + sub + 16 * e);
            }
      } else {
#pragma unroll
        for (int sq = 0; sq < 8; ++sq)
#pragma unroll
          for (int sub = 0; sub < 2; ++sub)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int jj = 16 * sq + 8 * sub + 2 * c + e;
              word |= ((sgn[t * 4 + (jj >> 5)] >> (jj & 31)) & 1u) << (2 * sq + sub + 16 * e);
            }
      }
      kw[w] = word;
    }
    uint32_t* nw = reinterpret_cast<uint32_t*>(page + pl.norms_off);
    for (int t = tid; t < kPage; t += kTcThreads) nw[t] = norms[t];
    uint32_t* vw = reinterpret_cast<uint32_t*>(page + pl.vbits_off);
    if (vb == 2) {
      for (int w = tid; w < 4 * (D / 16) * 32; w += kTcThreads) {
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
              word |= (uint32_t)vcode[t * D + 16 * mt + 8 * (rg & 1) + g] << (16 * e + 2 * vfield2(kap, rg));
            }
        vw[w] = word;
      }
    } else {
      for (int w = tid; w < 4 * (D / 16) * 32 * 2; w += kTcThreads) {
        const int kap = w & 1, ln = (w >> 1) & 31, mt = (w >> 6) % (D / 16), blk = w / (64 * (D / 16));
        const int g = ln >> 2, c = ln & 3;
        uint32_t word = 0;
#pragma unroll
        for (int rg = 0; rg < 4; ++rg)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int t = 32 * blk + 16 * kap + 8 * (rg >> 1) + 2 * c + e;
            word |= (uint32_t)vcode[t * D + 16 * mt + 8 * (rg & 1) + g] << (16 * e + 4 * vfield4(rg));
          }
        vw[w] = word;
      }
    }
    uint16_t* sw = reinterpret_cast<uint16_t*>(page + pl.vscale_off);
    for (int i = tid; i < kPage * (D / 32); i += kTcThreads) sw[vscale_idx(D, i / (D / 32), i % (D / 32))] = scales[i];
    __syncthreads();  // shared buffers are reused by the next page
  }
  if (!ok && tid == 0) set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;\n" ::"r"(tmem) : "memory");
}

// Ring update after the quantise launch: write the new ring tail and the sequence state.
// Dependents (the decode of this layer) are released only after the state is written: they read the
// sequence state before their own griddepcontrol.wait to start fetching pages early.
__global__ void __launch_bounds__(256) k_ring_update(AppendArgs a) {
  const int b = blockIdx.x;
  pdl_wait();  // the quantise launch has read the old ring and state
  const LayerView& lv = a.lv;
  const int slot = a.seq_ids[b];
  if (slot < 0 || slot >= lv.max_seqs) return;
  const int L = lv.state[2 * slot], F = lv.state[2 * slot + 1];
  const int Np = L > 0 ? kPage * ((L - 1) / kPage) : 0;
  if (a.flush) {
    __syncthreads();
    if (threadIdx.x == 0) {
      lv.state[2 * slot + 1] = L - Np;
      __threadfence();
    }
    __syncthreads();
    pdl_launch();
    return;
  }
  const int nn = a.n_new[b];
  const int L2 = L + nn;
  if (nn < 0 || nn > a.max_new || L2 > lv.max_ctx) return;
  const int Np2 = L2 > 0 ? kPage * ((L2 - 1) / kPage) : 0;
  const int p0 = max(L, Np2);
  const int d = lv.d, q4 = d / 4;
  const int n_items = (L2 - p0) * lv.Hkv * 2 * q4;  // (pos, head, which, quad)
  for (int it = threadIdx.x; it < n_items; it += blockDim.x) {
    const int quad = it % q4;
    int rest = it / q4;
    const int which = rest % 2;
    rest /= 2;
    const int hh = rest % lv.Hkv;
    const int pos = p0 + rest / lv.Hkv;
    const size_t src = (((size_t)b * a.max_new + (pos - L)) * lv.Hkv + hh) * d + 4 * quad;
    uint16_t* dst = lv.ring + ((((size_t)slot * lv.Hkv + hh) * 2 + which) * kPage + (pos - Np2)) * d + 4 * quad;
    const void* base = which ? a.v : a.k;
    uint2 out;
    if (a.dt == 0) {
      out = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + src);
    } else {
      const float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + src);
      out.x = (uint32_t)f32_to_bf16_rn(f.x) | ((uint32_t)f32_to_bf16_rn(f.y) << 16);
      out.y = (uint32_t)f32_to_bf16_rn(f.z) | ((uint32_t)f32_to_bf16_rn(f.w) << 16);
    }
    *reinterpret_cast<uint2*>(dst) = out;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    lv.state[2 * slot] = L2;
    lv.state[2 * slot + 1] = Np2 > Np ? 0 : F;
    __threadfence();
  }
  __syncthreads();
  pdl_launch();
}

__global__ void k_reset(int32_t* state_base, int n_layers, int max_seqs, int layer, const int32_t* seq_ids,
                        int batch) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int slot = seq_ids[b];
  if (slot < 0 || slot >= max_seqs) return;
  for (int l = 0; l < n_layers; ++l) {
    if (layer >= 0 && l != layer) continue;
    state_base[((size_t)l * max_seqs + slot) * 2] = 0;
    state_base[((size_t)l * max_seqs + slot) * 2 + 1] = 0;
  }
}

template <int D>
size_t quantize_smem_bytes() {
  return 2 * D * D + 2 * kPage * D + 4 * kPage + 2 * kPage * (D / 32) + 4 * 8 * D;
}

template <int D>
cudaError_t launch_quantize_d(const AppendArgs& a, int batch, int pages, cudaStream_t s) {
  const size_t smem = quantize_smem_bytes<D>();
  static bool attr_set = false;  // set once, outside any stream capture that follows
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_quantize_pages<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(batch, a.lv.Hkv, pages);
  return launch_pdl(k_quantize_pages<D>, grid, dim3(kQThreads), smem, s, a);
}

template <int D>
cudaError_t launch_append_small_d(const AppendArgs& a, int batch, size_t smem, cudaStream_t s) {
  static bool attr_set = false;  // set once, outside any stream capture that follows
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_append_small<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(k_append_small<D>, dim3(batch, a.lv.Hkv), dim3(kQThreads), smem, s, a);
}

cudaError_t launch_quantize(const AppendArgs& a, int batch, int pages, cudaStream_t s) {
  if (a.lv.d == 128) return launch_quantize_d<128>(a, batch, pages, s);
  return launch_quantize_d<256>(a, batch, pages, s);
}

// Bulk appends of head_dim 128 use the tcgen05 kernel: one persistent CTA per SM over all pages.
cudaError_t launch_quantize_bulk128(const AppendArgs& a, int batch, int pages, int sms, cudaStream_t s) {
  static bool attr_set = false;  // set once, outside any stream capture that follows
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_quantize_bulk128, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int ntasks = batch * a.lv.Hkv * pages;
  const int grid = std::max(1, std::min(ntasks, sms));
  return launch_pdl(k_quantize_bulk128, dim3(grid), dim3(kTcThreads), kTcSmem, s, a, pages, batch);
}

}  // namespace

cudaError_t launch_append(const tq_ctx* ctx, int layer, const void* k, const void* v, int dt,
                          const int32_t* seq_ids, const int32_t* n_new, int batch, int max_new, cudaStream_t s) {
  AppendArgs a;
  a.lv = layer_view(ctx, layer);
  a.k = k;
  a.v = v;
  a.dt = dt;
  a.seq_ids = seq_ids;
  a.n_new = n_new;
  a.max_new = max_new;
  a.flush = 0;
  if (max_new < kPage) {  // decode-sized appends: one launch (page on ring overflow + ring rows + state)
    const size_t smem = a.lv.d == 128 ? quantize_smem_bytes<128>() : quantize_smem_bytes<256>();
    return a.lv.d == 128 ? launch_append_small_d<128>(a, batch, smem, s) : launch_append_small_d<256>(a, batch, smem, s);
  }
  const int pages = (max_new + kPage - 1) / kPage;
  cudaError_t e = (a.lv.d == 128 && max_new >= kPage)
                      ? launch_quantize_bulk128(a, batch, pages, ctx->sm_count > 0 ? ctx->sm_count : 152, s)
                      : launch_quantize(a, batch, pages, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_ring_update, dim3(batch), dim3(256), 0, s, a);
}

cudaError_t launch_flush(const tq_ctx* ctx, int layer, const int32_t* seq_ids, int batch, cudaStream_t s) {
  AppendArgs a;
  a.lv = layer_view(ctx, layer);
  a.k = a.v = nullptr;
  a.dt = 0;
  a.seq_ids = seq_ids;
  a.n_new = nullptr;
  a.max_new = 0;
  a.flush = 1;
  cudaError_t e = launch_quantize(a, batch, 1, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_ring_update, dim3(batch), dim3(32), 0, s, a);
}

cudaError_t launch_reset(const tq_ctx* ctx, int layer, const int32_t* seq_ids, int batch, cudaStream_t s) {
  const LayerView lv = layer_view(ctx, 0);
  k_reset<<<(batch + 127) / 128, 128, 0, s>>>(lv.state, ctx->cfg.n_layers, ctx->cfg.max_seqs, layer, seq_ids, batch);
  return cudaGetLastError();
}

}  // namespace tq
