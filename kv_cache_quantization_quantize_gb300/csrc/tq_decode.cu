// Hybrid decode attention ([Guide] §五.1 and §七): split-K flash decoding over the packed history
// plus one exact split over the bf16 ring, then an exact log-sum-exp merge.
//
// Scores. For a packed token (n, idx, gamma, sign) and query head q:
//   s = scale * n * ( <Pi q, c[idx]> + sqrt(pi/2)/d * gamma * <S Pi q, 2 sign - 1> )  ([Guide] §二, TurboQuantProd).
// The 2-bit codebook is odd-symmetric, so c[idx] = alpha*(2 b_hi - 1) + beta*(2 b_lo - 1), with
// alpha = (c2+c3)/2 and beta = (c3-c2)/2. Each score is therefore a sum of three bit-plane dot
// products.
//   - They run on fp8 tensor cores (mma.sync m16n8k32 e4m3). Operand A = 4 fp8 limbs of the scaled
//     query for up to 4 heads (16 rows). Operand B = key bits masked straight out of the packed
//     words; each byte is 0 or a power of two.
//   - The powers of two are undone by prescaling A.
// Values. Code fields are masked into f16 subnormals code * 2^(pos-24) and multiplied (mma.sync
// m16n8k16) by P' = p * s * 2^(24-pos). The mid-rise offset (2^(b-1) - 1/2) * sum(p*s) is removed at
// the end of the split.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>

#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kDThreads = 128;  // 4 warps; warp w owns tokens 32w..32w+31 of every page

struct DecodeArgs {
  LayerView lv;
  const uint16_t* q;  // bf16 [B][Hq][D]
  float* out;         // [B][Hq][D]
  const int32_t* seq_ids;
  float scale;
  uint8_t* ws;
  DecodePlan plan;
};

// e4m3 value of bit position p (0..5) of a byte: mantissa bits give subnormals 2^-9, 2^-8, 2^-7;
// exponent bits 3, 4, 5 give 2^-6, 2^-5, 2^-3.
__host__ __device__ __forceinline__ int e4m3_bit_exp(int p) {
  return p == 0 ? -9 : p == 1 ? -8 : p == 2 ? -7 : p == 3 ? -6 : p == 4 ? -5 : -3;
}

__device__ __forceinline__ void mma_e4m3(float (&c)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ---- mbarrier / bulk copy (async proxy) ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bounded wait on an mbarrier phase: returns false after ~2^22 polls (seconds), never hangs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void seq_packed(const LayerView& lv, int slot, int& L, int& Np, int& P) {
  L = lv.state[2 * slot];
  const int F = lv.state[2 * slot + 1];
  Np = L > 0 ? kPage * ((L - 1) / kPage) : 0;
  P = Np + F;
}

// =============================================================================================
// Query prep: q_rot = Pi q, q_proj = S q_rot; fp8 limbs of the three bit-plane operands
// =============================================================================================
template <int D>
__global__ void __launch_bounds__(kDThreads) k_prep(DecodeArgs a) {
  constexpr int NE = D / 32;
  constexpr int KST = 3 * D / 32;  // k-steps of 32 coordinates over the three planes
  __shared__ float qr[kMaxG][D];
  __shared__ float qp[kMaxG][D];
  __shared__ float red[kMaxG][4];
  const int b = blockIdx.x, h = blockIdx.y;
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = lv.G;
  // warp w rotates head w (zero rows for heads >= G)
  {
    float x[NE];
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const int j = (e >> 2) * 128 + 4 * lane + (e & 3);
      float qv = 0.f;
      if (warp < G) qv = bf16_to_f32(a.q[((size_t)b * lv.Hq + h * G + warp) * D + j]);
      x[e] = qv * lv.D[j];
    }
    warp_fwht<NE>(x, lane);
    const float s = rsqrtf((float)D);
#pragma unroll
    for (int e = 0; e < NE; ++e) qr[warp][(e >> 2) * 128 + 4 * lane + (e & 3)] = x[e] * s;
  }
  __syncthreads();
  // q_proj[i] = sum_j S[i][j] q_rot[j] = sum_j St[j][i] q_rot[j]
  for (int i = tid; i < D; i += kDThreads) {
    float acc[kMaxG] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < D; ++j) {
      const float sv = bf16_to_f32(lv.St[(size_t)j * D + i]);
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) acc[g] = fmaf(sv, qr[g][j], acc[g]);
    }
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) qp[g][i] = acc[g];
  }
  __syncthreads();
  const float alpha2 = 2.f * lv.cb[8], beta2 = 2.f * lv.cb[9];
  // per-head power-of-two scales: largest prescaled operand magnitude in [128, 256) (e4m3 max 448)
  if (warp < kMaxG) {
    float mm = 0.f, mq = 0.f;
    for (int j = lane; j < D; j += 32) {
      const int jj = j & 127, ks = jj >> 5, hb = (jj >> 4) & 1;
      int p = 2 * ks + hb;
      p = p < 6 ? p : p - 2;
      const float pre = exp2f((float)-e4m3_bit_exp(p));
      mm = fmaxf(mm, fabsf(alpha2 * qr[warp][j]) * pre);
      mq = fmaxf(mq, fabsf(2.f * qp[warp][j]) * pre);
    }
    mm = warp_max(mm);
    mq = warp_max(mq);
    if (lane == 0) {
      red[warp][0] = mm > 0.f ? exp2f(floorf(log2f(256.f / mm))) : 1.f;
      red[warp][1] = mq > 0.f ? exp2f(floorf(log2f(256.f / mq))) : 1.f;
    }
  }
  __syncthreads();
  // fragments: frag[kidx][lane] = 4 u32 (16 fp8); row = 4*limb + head
  uint8_t* prep = a.ws + a.plan.prep_off + ((size_t)b * lv.Hkv + h) * a.plan.prep_stride;
  uint32_t* frag = reinterpret_cast<uint32_t*>(prep);
  float* cst = reinterpret_cast<float*>(prep + (size_t)KST * 32 * 16);
  float csum_m[kMaxG] = {0, 0, 0, 0}, csum_q[kMaxG] = {0, 0, 0, 0};
  for (int item = tid; item < KST * 32; item += kDThreads) {
    const int kidx = item / 32, ln = item % 32;
    const int g = ln >> 2, c = ln & 3;
    const int pi = kidx / (D / 32), loc = kidx % (D / 32), half = loc / 4, ks = loc % 4;
    uint32_t regs[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = g + 8 * (r & 1);
      const int limb = row >> 2, head = row & 3;
      uint32_t word = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = 4 * c + i + 16 * (r >> 1);
        const int j = 128 * half + 32 * ks + k;
        int p = 2 * ks + (k >> 4);
        p = p < 6 ? p : p - 2;
        const float pre = exp2f((float)-e4m3_bit_exp(p));
        const float base = pi == 0 ? alpha2 * qr[head][j] : pi == 1 ? beta2 * qr[head][j] : 2.f * qp[head][j];
        const float lam = pi < 2 ? red[head][0] : red[head][1];
        float x = base * lam * pre;
        float limb_v = 0.f;
        __nv_fp8_e4m3 f8;
        for (int l = 0; l <= limb; ++l) {
          f8 = __nv_fp8_e4m3(x);
          limb_v = float(f8);
          x -= limb_v;
        }
        word |= (uint32_t)f8.__x << (8 * i);
        // represented operand value (sum of limbs) times the bit weight 2^e, for the offset constants
        if (limb == 0) {
          float xx = base * lam * pre, rep = 0.f;
          for (int l = 0; l < 4; ++l) {
            const __nv_fp8_e4m3 t8(xx);
            rep += float(t8);
            xx -= float(t8);
          }
          const float w = rep * exp2f((float)e4m3_bit_exp(p));
          if (pi < 2) csum_m[head] += w; else csum_q[head] += w;
        }
      }
      regs[r] = word;
    }
    reinterpret_cast<uint4*>(frag)[item] = make_uint4(regs[0], regs[1], regs[2], regs[3]);
  }
  // reduce the offset constants over the block
  __syncthreads();
  __shared__ float cs[2][kMaxG];
  if (tid < 2 * kMaxG) cs[tid / kMaxG][tid % kMaxG] = 0.f;
  __syncthreads();
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) {
    const float vm = warp_sum(csum_m[g]), vq = warp_sum(csum_q[g]);
    if (lane == 0) {
      atomicAdd(&cs[0][g], vm);
      atomicAdd(&cs[1][g], vq);
    }
  }
  __syncthreads();
  if (tid < kMaxG) {
    const float kappa = 1.2533141373155003f / (float)D;  // sqrt(pi/2) / d
    cst[4 * tid + 0] = a.scale * kLog2e / red[tid][0];
    cst[4 * tid + 1] = 0.5f * cs[0][tid];
    cst[4 * tid + 2] = a.scale * kLog2e * kappa / red[tid][1];
    cst[4 * tid + 3] = 0.5f * cs[1][tid];
  }
}

// =============================================================================================
// Split-K decode over packed pages (blockIdx.x < n_splits) and the exact ring split (== n_splits)
// =============================================================================================
template <int D>
__device__ void ring_split(const DecodeArgs& a, int b, int h, int slot, float* part, uint8_t* smem_raw) {
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x;
  int L, Np, P;
  seq_packed(lv, slot, L, Np, P);
  const int F = P - Np, R = L - Np;
  float* qs = reinterpret_cast<float*>(smem_raw);        // [4][D]
  float* sc = qs + kMaxG * D;                             // [4][128]
  float* red = sc + kMaxG * kPage;                        // [4][4] scratch
  const int G = lv.G;
  for (int i = tid; i < kMaxG * D; i += kDThreads) {
    const int g = i / D, j = i % D;
    qs[i] = g < G ? bf16_to_f32(a.q[((size_t)b * lv.Hq + h * G + g) * D + j]) : 0.f;
  }
  __syncthreads();
  const uint16_t* rk = lv.ring + (((size_t)slot * lv.Hkv + h) * 2 + 0) * kPage * D;
  const uint16_t* rv = rk + (size_t)kPage * D;
  const float s2 = a.scale * kLog2e;
  {
    const int i = F + tid;
    float acc[kMaxG] = {0.f, 0.f, 0.f, 0.f};
    if (i < R) {
      const uint2* row = reinterpret_cast<const uint2*>(rk + (size_t)i * D);
      for (int q4 = 0; q4 < D / 4; ++q4) {
        const uint2 u = row[q4];
        const float k0 = __uint_as_float(u.x << 16), k1 = __uint_as_float(u.x & 0xffff0000u);
        const float k2 = __uint_as_float(u.y << 16), k3 = __uint_as_float(u.y & 0xffff0000u);
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) {
          const float* qq = qs + g * D + 4 * q4;
          acc[g] = fmaf(qq[0], k0, fmaf(qq[1], k1, fmaf(qq[2], k2, fmaf(qq[3], k3, acc[g]))));
        }
      }
    }
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) sc[g * kPage + tid] = i < R ? acc[g] * s2 : -INFINITY;
  }
  __syncthreads();
  const int lane = tid & 31, warp = tid >> 5;
  // warp g reduces head g: max and sum of exp2
  {
    float m = -INFINITY;
    for (int t = lane; t < kPage; t += 32) m = fmaxf(m, sc[warp * kPage + t]);
    m = warp_max(m);
    float l = 0.f;
    for (int t = lane; t < kPage; t += 32) {
      const float s = sc[warp * kPage + t];
      const float p = s == -INFINITY ? 0.f : exp2f(s - m);
      sc[warp * kPage + t] = p;
      l += p;
    }
    l = warp_sum(l);
    if (lane == 0) {
      red[warp * 4 + 0] = m;
      red[warp * 4 + 1] = l;
    }
  }
  __syncthreads();
  for (int j = tid; j < D; j += kDThreads) {
    float o[kMaxG] = {0.f, 0.f, 0.f, 0.f};
    for (int i = F; i < R; ++i) {
      const float vv = bf16_to_f32(rv[(size_t)i * D + j]);
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) o[g] = fmaf(sc[g * kPage + (i - F)], vv, o[g]);
    }
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) part[2 * kMaxG + g * D + j] = o[g];
  }
  if (tid < kMaxG) {
    part[tid] = red[tid * 4 + 0];
    part[kMaxG + tid] = red[tid * 4 + 1];
  }
}

template <int D, int VB, int STAGES>
__global__ void __launch_bounds__(kDThreads) k_decode(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const LayerView& lv = a.lv;
  const int sp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nsp = a.plan.n_splits;
  float* part = reinterpret_cast<float*>(a.ws + a.plan.part_off +
                                         (((size_t)b * lv.Hkv + h) * (nsp + 1) + sp) * a.plan.part_stride);
  const int slot = a.seq_ids[b];
  if (slot < 0 || slot >= lv.max_seqs) {
    if (tid < kMaxG) {
      part[tid] = -INFINITY;
      part[kMaxG + tid] = 0.f;
    }
    return;
  }
  if (sp == nsp) {
    ring_split<D>(a, b, h, slot, part, smem);
    return;
  }
  int L, Np, P;
  seq_packed(lv, slot, L, Np, P);
  const int n_pages = (P + kPage - 1) / kPage;
  const int pps = a.plan.pages_per_split;
  if (sp == 0 && tid == 0 && n_pages > nsp * pps) set_status(lv.status, TQ_DEV_ERR_SPLITS);
  const int pg0 = sp * pps, pg1 = min(n_pages, pg0 + pps);
  if (pg0 >= pg1) {
    if (tid < kMaxG) {
      part[tid] = -INFINITY;
      part[kMaxG + tid] = 0.f;
    }
    return;
  }
  const PageLayout pl = page_layout(D, VB);
  const uint32_t PB = pl.bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint8_t* stage0 = smem + 128;
  const uint8_t* gpages = lv.pages + ((size_t)slot * lv.Hkv + h) * lv.max_pages * PB;
  const int npg = pg1 - pg0;
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    for (int s = 0; s < STAGES && s < npg; ++s) {
      mbar_expect_tx(&full[s], PB);
      bulk_g2s(stage0 + (size_t)s * PB, gpages + (size_t)(pg0 + s) * PB, PB, &full[s]);
    }
  }
  // score operand A (q limbs) and per-head constants
  constexpr int KST = 3 * D / 32;
  constexpr int HALVES = D / 128;
  const uint8_t* prep = a.ws + a.plan.prep_off + ((size_t)b * lv.Hkv + h) * a.plan.prep_stride;
  uint4 af[KST];
#pragma unroll
  for (int k = 0; k < KST; ++k) af[k] = reinterpret_cast<const uint4*>(prep)[k * 32 + lane];
  const int g = lane >> 2, c = lane & 3, hh = g & 3;
  const float* cst = reinterpret_cast<const float*>(prep + (size_t)KST * 32 * 16);
  const float u_m = cst[4 * hh + 0], c_m = cst[4 * hh + 1], u_q = cst[4 * hh + 2], c_q = cst[4 * hh + 3];
  const bool live_col = g < lv.G;  // B columns >= G (padding heads) are zero
  constexpr int NG = D / 32;       // value groups
  constexpr int NMT = D / 16;      // m-tiles of the value accumulator
  float O[NMT][4];
#pragma unroll
  for (int mt = 0; mt < NMT; ++mt) O[mt][0] = O[mt][1] = O[mt][2] = O[mt][3] = 0.f;
  float m_eff = -INFINITY, l_acc = 0.f;
  float lg[NG];
#pragma unroll
  for (int q = 0; q < NG; ++q) lg[q] = 0.f;
  __syncthreads();
  bool timed_out = false;

  for (int ip = 0; ip < npg; ++ip) {
    const int s = ip % STAGES;
    if (!mbar_wait(&full[s], (ip / STAGES) & 1)) {
      timed_out = true;
      break;
    }
    const uint8_t* pg = stage0 + (size_t)s * PB;
    const int valid = min(kPage, P - (pg0 + ip) * kPage);
    const uint32_t* kw = reinterpret_cast<const uint32_t*>(pg + pl.kbits_off);
    // ---- scores of the warp's 32 tokens (4 n-tiles of 8) ----
    float sc[4][2];
#pragma unroll
    for (int ntl = 0; ntl < 4; ++ntl) {
      const int nt = 4 * warp + ntl;
      float am[4] = {0.f, 0.f, 0.f, 0.f}, aq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int pi = 0; pi < 3; ++pi) {
#pragma unroll
        for (int hf = 0; hf < HALVES; ++hf) {
          const uint32_t w = kw[((nt * 3 + pi) * HALVES + hf) * 32 + lane];
          const uint32_t ws = w >> 2;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t b0 = ks < 3 ? (w & (0x01010101u << (2 * ks))) : (ws & 0x10101010u);
            const uint32_t b1 = ks < 3 ? (w & (0x02020202u << (2 * ks))) : (ws & 0x20202020u);
            const int kidx = pi * (D / 32) + hf * 4 + ks;
            if (pi < 2) mma_e4m3(am, af[kidx], b0, b1);
            else mma_e4m3(aq, af[kidx], b0, b1);
          }
        }
      }
      float m0 = am[0] + am[2], m1 = am[1] + am[3];
      float q0 = aq[0] + aq[2], q1 = aq[1] + aq[3];
      m0 += __shfl_xor_sync(0xffffffffu, m0, 16);
      m1 += __shfl_xor_sync(0xffffffffu, m1, 16);
      q0 += __shfl_xor_sync(0xffffffffu, q0, 16);
      q1 += __shfl_xor_sync(0xffffffffu, q1, 16);
      const int t0 = 8 * nt + 2 * c;
      const uint2 nr = *reinterpret_cast<const uint2*>(pg + pl.norms_off + 4 * t0);
      const float n0 = __half2float(__ushort_as_half((uint16_t)(nr.x & 0xffff)));
      const float g0 = __half2float(__ushort_as_half((uint16_t)(nr.x >> 16)));
      const float n1 = __half2float(__ushort_as_half((uint16_t)(nr.y & 0xffff)));
      const float g1 = __half2float(__ushort_as_half((uint16_t)(nr.y >> 16)));
      sc[ntl][0] = t0 < valid ? n0 * fmaf(u_m, m0 - c_m, u_q * g0 * (q0 - c_q)) : -INFINITY;
      sc[ntl][1] = t0 + 1 < valid ? n1 * fmaf(u_m, m1 - c_m, u_q * g1 * (q1 - c_q)) : -INFINITY;
    }
    // ---- largest value scale among the warp's 32 tokens ----
    const uint16_t* vsc = reinterpret_cast<const uint16_t*>(pg + pl.vscale_off);
    float smax = 0.f;
    {
      const uint16_t* row = vsc + (32 * warp + lane) * NG;
#pragma unroll
      for (int q = 0; q < NG; ++q) smax = fmaxf(smax, __half2float(__ushort_as_half(row[q])));
    }
    smax = warp_max(smax);
    // ---- online softmax in exp2 units; m_eff also keeps P' = p * s * 2^24 inside f16 range ----
    float mx = -INFINITY;
#pragma unroll
    for (int ntl = 0; ntl < 4; ++ntl) mx = fmaxf(mx, fmaxf(sc[ntl][0], sc[ntl][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    int e2 = 0;
    frexpf(smax, &e2);
    const float E = smax > 0.f ? (float)(9 + e2) : 0.f;
    const float m_new = fmaxf(m_eff, mx + E);
    const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_eff - m_new);
    m_eff = m_new;
    l_acc *= alpha;
#pragma unroll
    for (int q = 0; q < NG; ++q) lg[q] *= alpha;
    const float aA = __shfl_sync(0xffffffffu, alpha, (8 * c) & 31);
    const float aB = __shfl_sync(0xffffffffu, alpha, (8 * c + 4) & 31);
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) {
      O[mt][0] *= aA;
      O[mt][1] *= aB;
      O[mt][2] *= aA;
      O[mt][3] *= aB;
    }
    float p[4][2];
#pragma unroll
    for (int ntl = 0; ntl < 4; ++ntl)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float x = sc[ntl][e];
        p[ntl][e] = (x == -INFINITY || !live_col) ? 0.f : exp2f(x - m_eff);
        l_acc += p[ntl][e];
      }
    // ---- P.V on f16 tensor cores, one value group (two m-tiles) at a time ----
    const uint32_t* vw = reinterpret_cast<const uint32_t*>(pg + pl.vbits_off);
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      uint32_t bf[2][2];
#pragma unroll
      for (int kap = 0; kap < 2; ++kap)
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          const int ntl = 2 * kap + hi;
          const int t0 = 8 * (4 * warp + ntl) + 2 * c;
          const float s0 = __half2float(__ushort_as_half(vsc[t0 * NG + q]));
          const float s1 = __half2float(__ushort_as_half(vsc[(t0 + 1) * NG + q]));
          const int pos = VB == 2 ? vpos2(kap, hi) : vpos4(hi);
          const float pre = (float)(1u << (24 - pos));
          bf[kap][hi] = pack_half2(p[ntl][0] * s0 * pre, p[ntl][1] * s1 * pre);
          // the mid-rise offset is removed with the same f16-rounded weights the MMA multiplies
          const float2 wr = __half22float2(*reinterpret_cast<const __half2*>(&bf[kap][hi]));
          lg[q] = fmaf(wr.x + wr.y, 1.0f / pre, lg[q]);
        }
#pragma unroll
      for (int mh = 0; mh < 2; ++mh) {
        const int mt = 2 * q + mh;
        if (VB == 2) {
          const uint32_t w = vw[(warp * NMT + mt) * 32 + lane];
          const uint32_t w2 = w >> 2, w6 = w >> 6;
          mma_f16(O[mt], w & 0x00030003u, w2 & 0x00030003u, w & 0x00300030u, w6 & 0x00300030u, bf[0][0], bf[0][1]);
          mma_f16(O[mt], w & 0x00C000C0u, w6 & 0x00C000C0u, w & 0x03000300u, w6 & 0x03000300u, bf[1][0], bf[1][1]);
        } else {
          const uint2 ww = reinterpret_cast<const uint2*>(vw)[(warp * NMT + mt) * 32 + lane];
          const uint32_t x0 = ww.x, x8 = ww.x >> 8, y0 = ww.y, y8 = ww.y >> 8;
          mma_f16(O[mt], x0 & 0x000F000Fu, x8 & 0x000F000Fu, x0 & 0x00F000F0u, x8 & 0x00F000F0u, bf[0][0], bf[0][1]);
          mma_f16(O[mt], y0 & 0x000F000Fu, y8 & 0x000F000Fu, y0 & 0x00F000F0u, y8 & 0x00F000F0u, bf[1][0], bf[1][1]);
        }
      }
    }
    __syncthreads();  // every warp is done with stage s
    if (tid == 0 && ip + STAGES < npg) {
      mbar_expect_tx(&full[s], PB);
      bulk_g2s(stage0 + (size_t)s * PB, gpages + (size_t)(pg0 + ip + STAGES) * PB, PB, &full[s]);
    }
  }
  if (timed_out) {
    if (tid == 0) set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
  }
  // ---- merge the four warps' partials through shared memory ----
  __syncthreads();
  float* wm = reinterpret_cast<float*>(stage0);   // [4 warps][4 heads]
  float* wl = wm + 16;                            // [4][4]
  float* wlg = wl + 16;                           // [4][4][NG]
  float* wo = wlg + 16 * NG;                      // [4][4][D]
  {
    float l = l_acc;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      lg[q] += __shfl_xor_sync(0xffffffffu, lg[q], 1);
      lg[q] += __shfl_xor_sync(0xffffffffu, lg[q], 2);
    }
    if (c == 0 && g < kMaxG) {
      wm[warp * 4 + g] = m_eff;
      wl[warp * 4 + g] = l;
#pragma unroll
      for (int q = 0; q < NG; ++q) wlg[(warp * 4 + g) * NG + q] = lg[q];
    }
    if (c < 2) {
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) {
        const int j0 = 16 * mt + g;
        wo[(warp * 4 + 2 * c) * D + j0] = O[mt][0];
        wo[(warp * 4 + 2 * c + 1) * D + j0] = O[mt][1];
        wo[(warp * 4 + 2 * c) * D + j0 + 8] = O[mt][2];
        wo[(warp * 4 + 2 * c + 1) * D + j0 + 8] = O[mt][3];
      }
    }
  }
  __syncthreads();
  const float off = (float)(1 << (VB - 1)) - 0.5f;
  for (int i = tid; i < kMaxG * D; i += kDThreads) {
    const int hd = i / D, j = i % D;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) m = fmaxf(m, wm[w * 4 + hd]);
    float o = 0.f, l = 0.f;
    if (m != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = wm[w * 4 + hd];
        const float f = mw == -INFINITY ? 0.f : exp2f(mw - m);
        o += f * (wo[(w * 4 + hd) * D + j] - off * wlg[(w * 4 + hd) * NG + j / 32]);
        l += f * wl[w * 4 + hd];
      }
    }
    part[2 * kMaxG + hd * D + j] = o;
    if (j == 0) {
      part[hd] = m;
      part[kMaxG + hd] = l;
    }
  }
}

// =============================================================================================
// Combine: LSE merge of history splits (rotated basis) -> Pi^T -> exact merge with the ring split
// =============================================================================================
template <int D>
__global__ void __launch_bounds__(kDThreads) k_combine(DecodeArgs a) {
  constexpr int NE = D / 32;
  const LayerView& lv = a.lv;
  const int b = blockIdx.x, h = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;  // warp = query head within the group
  if (warp >= lv.G) return;
  const int nsp = a.plan.n_splits;
  const uint8_t* base = a.ws + a.plan.part_off + ((size_t)b * lv.Hkv + h) * (nsp + 1) * a.plan.part_stride;
  float m = -INFINITY;
  for (int s = 0; s < nsp; ++s) m = fmaxf(m, reinterpret_cast<const float*>(base + s * a.plan.part_stride)[warp]);
  float o[NE];
#pragma unroll
  for (int e = 0; e < NE; ++e) o[e] = 0.f;
  float l = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < nsp; ++s) {
      const float* pt = reinterpret_cast<const float*>(base + s * a.plan.part_stride);
      const float ms = pt[warp];
      if (ms == -INFINITY) continue;
      const float f = exp2f(ms - m);
      l = fmaf(f, pt[kMaxG + warp], l);
#pragma unroll
      for (int hf = 0; hf < NE / 4; ++hf) {
        const float4 v = *reinterpret_cast<const float4*>(pt + 2 * kMaxG + warp * D + 128 * hf + 4 * lane);
        o[4 * hf + 0] = fmaf(f, v.x, o[4 * hf + 0]);
        o[4 * hf + 1] = fmaf(f, v.y, o[4 * hf + 1]);
        o[4 * hf + 2] = fmaf(f, v.z, o[4 * hf + 2]);
        o[4 * hf + 3] = fmaf(f, v.w, o[4 * hf + 3]);
      }
    }
  }
  // Pi^T o = D * (H o) / sqrt(d)
  warp_fwht<NE>(o, lane);
  const float rs = rsqrtf((float)D);
#pragma unroll
  for (int e = 0; e < NE; ++e) o[e] *= rs * lv.D[(e >> 2) * 128 + 4 * lane + (e & 3)];
  const float* rp = reinterpret_cast<const float*>(base + nsp * a.plan.part_stride);
  const float mr = rp[warp], lr = rp[kMaxG + warp];
  const float mm = fmaxf(m, mr);
  const float fh = (m == -INFINITY) ? 0.f : exp2f(m - mm);
  const float fr = (mr == -INFINITY) ? 0.f : exp2f(mr - mm);
  const float den = fh * l + fr * lr;
  const float inv = den > 0.f ? 1.f / den : 0.f;
  float* out = a.out + ((size_t)b * lv.Hq + h * lv.G + warp) * D;
#pragma unroll
  for (int hf = 0; hf < NE / 4; ++hf) {
    const float4 rv = *reinterpret_cast<const float4*>(rp + 2 * kMaxG + warp * D + 128 * hf + 4 * lane);
    float4 r;
    r.x = (fh * o[4 * hf + 0] + fr * rv.x) * inv;
    r.y = (fh * o[4 * hf + 1] + fr * rv.y) * inv;
    r.z = (fh * o[4 * hf + 2] + fr * rv.z) * inv;
    r.w = (fh * o[4 * hf + 3] + fr * rv.w) * inv;
    *reinterpret_cast<float4*>(out + 128 * hf + 4 * lane) = r;
  }
}

template <int D, int VB>
cudaError_t launch_decode_dv(const DecodeArgs& a, int batch, int phase, cudaStream_t s) {
  constexpr int STAGES = D == 128 ? 4 : 3;
  const PageLayout pl = page_layout(D, VB);
  const size_t merge_bytes = sizeof(float) * (16 + 16 + 16 * (D / 32) + 16 * D);
  const size_t ring_bytes = sizeof(float) * (kMaxG * D + kMaxG * kPage + 16);
  size_t smem = 128 + (size_t)STAGES * pl.bytes;
  smem = std::max(smem, 128 + merge_bytes);
  smem = std::max(smem, ring_bytes);
  static bool attr_set = false;  // set once, outside any stream capture that follows
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_decode<D, VB, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (phase < 0 || phase == 0) {
    k_prep<D><<<dim3(batch, a.lv.Hkv), kDThreads, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (phase < 0 || phase == 1) {
    k_decode<D, VB, STAGES><<<dim3(a.plan.n_splits + 1, a.lv.Hkv, batch), kDThreads, smem, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (phase < 0 || phase == 2) {
    k_combine<D><<<dim3(batch, a.lv.Hkv), kDThreads, 0, s>>>(a);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_decode(const tq_ctx* ctx, int layer, const void* q, float* out, const int32_t* seq_ids,
                          int batch, float scale, void* ws, const DecodePlan& plan, int phase, cudaStream_t s) {
  DecodeArgs a;
  a.lv = layer_view(ctx, layer);
  a.q = static_cast<const uint16_t*>(q);
  a.out = out;
  a.seq_ids = seq_ids;
  a.scale = scale;
  a.ws = static_cast<uint8_t*>(ws);
  a.plan = plan;
  const int d = ctx->cfg.head_dim, vb = ctx->cfg.value_bits;
  if (d == 128 && vb == 2) return launch_decode_dv<128, 2>(a, batch, phase, s);
  if (d == 128 && vb == 4) return launch_decode_dv<128, 4>(a, batch, phase, s);
  if (d == 256 && vb == 2) return launch_decode_dv<256, 2>(a, batch, phase, s);
  return launch_decode_dv<256, 4>(a, batch, phase, s);
}

}  // namespace tq

// =============================================================================================
// Decode without caller-provided scratch.
//
// Some callers cannot allocate device memory at the point where they decode. Examples:
//   - a host thread that runs inside a graph-building or real-time path, where cudaMalloc
//     (which can synchronise the device) is not allowed;
//   - an embedding runtime that owns all device memory and exposes no allocator;
//   - a plugin ABI that passes in only the tensors of the operation itself.
// For them this variant takes only inputs and outputs. Its scratch (query-prep operands and split
// partials) lives in the file-scope device array below, so it has a fixed maximum size.
// =============================================================================================
namespace tq {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB, held by every device that loads libtq
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. The first call on each device looks it
// up with cudaGetSymbolAddress; later calls reuse the cached address.
cudaError_t noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_decode_attention_noalloc(tq_ctx* ctx, int layer, const void* q, float* out,
                                                 const int32_t* d_seq_ids, int batch, float softmax_scale,
                                                 int max_ctx_hint, tq_stream_t stream) {
  tq_status st = tq::check_layer_ready(ctx, layer);
  if (st != TQ_OK) return st;
  if (batch < 0) return tq::set_error(TQ_ERR_INVALID_ARG, "batch is negative");
  if (batch == 0) return tq::set_error(TQ_OK, "");
  if (!q || !out || !d_seq_ids) return tq::set_error(TQ_ERR_INVALID_ARG, "NULL q/out/d_seq_ids");
  if (batch > ctx->cfg.max_seqs) return tq::set_error(TQ_ERR_CAPACITY, "batch > max_seqs");
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
    return tq::set_error(TQ_ERR_INVALID_ARG, "q/out must be 16-byte aligned");
  if (!(softmax_scale == softmax_scale)) return tq::set_error(TQ_ERR_INVALID_ARG, "softmax_scale is NaN");
  if (ctx->device >= tq::kMaxDevices) return tq::set_error(TQ_ERR_UNSUPPORTED, "device index >= 64");
  const tq::DecodePlan plan = tq::decode_plan(ctx, batch, max_ctx_hint);
  if (plan.bytes > tq::kNoAllocScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "decode scratch of %zu bytes exceeds the built-in %zu-byte scratch of tq_decode_attention_noalloc; "
             "lower batch or max_ctx_hint, or use tq_decode_attention with a caller workspace",
             plan.bytes, tq::kNoAllocScratchBytes);
    return tq::set_error(TQ_ERR_CAPACITY, msg);
  }
  void* scratch = nullptr;
  cudaError_t e = tq::noalloc_scratch(&scratch);
  if (e != cudaSuccess) return tq::set_error(TQ_ERR_CUDA, cudaGetErrorString(e));
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)ctx->cfg.head_dim);
  e = tq::launch_decode(ctx, layer, q, out, d_seq_ids, batch, scale, scratch, plan, -1, (cudaStream_t)stream);
  if (e != cudaSuccess) return tq::set_error(TQ_ERR_CUDA, cudaGetErrorString(e));
  return tq::set_error(TQ_OK, "");
}
