// Hybrid decode attention ([Guide] §五.1 and §七): split-K flash decoding over the packed history
// plus one exact split over the bf16 ring, then an exact log-sum-exp merge.
//
// Scores. For a packed token (n, idx, gamma, sign) and query head q:
//   s = scale * n * ( <Pi q, c[idx]> + sqrt(pi/2)/d * gamma * <S Pi q, 2 sign - 1> )  ([Guide] §二, TurboQuantProd).
// The codebook is odd-symmetric, so c[idx] is a weighted sum of +-1 bit planes:
//   - 2-bit index (key_bits 3): c = alpha (2 b1 - 1) + beta (2 b0 - 1), alpha = (c2+c3)/2, beta = (c3-c2)/2;
//   - 3-bit index (key_bits 4): c = A s2 + B t1 + C t0 + E s2 t1 t0 (s, t = 2 bit - 1), the last plane
//     being b2 ^ b1 ^ b0, with A, B, C, E fitted exactly to c4..c7.
// Each score is therefore a sum of bit-plane dot products (3 or 5) on f16 tensor cores (mma.sync m16n8k16):
//   - A = key bits masked straight out of the packed words. Bits 0..11 of an f16 half are exactly
//     2^(q-24) when set, and 0 otherwise.
//   - B = the query, prescaled by 2^(24-q), for up to 4 heads.
//   - The -1 of each +-1 plane is a per-head constant, subtracted once.
// Values. Code fields are masked into f16 subnormals code * 2^(pos-24) and multiplied (m16n8k16) by
// P' = p * s * 2^(24-pos). The mid-rise offset (2^(b-1) - 1/2) * sum(P') is removed at the end of
// the split, using the same f16 weights.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Wait-timeout test hook (tq_debug_decode_wait_fault), read by every decode launch.
std::atomic<int> g_fault_stage{-1};
std::atomic<int> g_fault_polls{0};

struct DecodeArgs {
  LayerView lv;
  int qpr;              // queries per cache row: 1 for decode; > 1 for prefill (row b = batch row b / qpr)
  const int32_t* n_q;   // prefill: queries of each batch row (its last n_q tokens); nullptr for decode
  const uint16_t* q;  // bf16 [B][Hq][D]
  float* out;         // [B][Hq][D]
  const int32_t* seq_ids;
  float scale;
  uint8_t* ws;
  DecodePlan plan;
  // Wait-timeout test hook (tq_debug_decode_wait_fault): >= 0 makes the first split CTA of (row 0, KV head 0)
  // leave page stage `fault_stage` of its first page stream without a copy; its wait on that stage gives up
  // after `fault_polls` polls. -1 in normal use.
  int fault_stage;
  uint32_t fault_polls;
};

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

// f16x2 pattern of -v * 2^(pos-24) in both halves (an f16 subnormal: v << pos with the sign bit).
__host__ __device__ constexpr uint32_t voff_pattern(uint32_t v, int pos) {
  return (0x8000u | (v << pos)) * 0x00010001u;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// ld.global.cg (L2 only: data written by other CTAs of this grid) that the compiler cannot move above
// a guard; __ldcg is a non-volatile asm and may be hoisted.
__device__ __forceinline__ float ld_cg_f(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];\n" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];\n" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ float2 ld_cg_f2(const float* p) {
  float2 v;
  asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "l"(p));
  return v;
}
// This lane's D / 32 values of a d-row in the lane_coord layout (L2 loads / plain stores).
template <int D>
__device__ __forceinline__ void ld_cg_row(const float* row, int lane, float (&x)[D / 32]) {
  if (D == 64) {
    const float2 v = ld_cg_f2(row + 2 * lane);
    x[0] = v.x;
    x[D / 32 - 1] = v.y;
  } else {
#pragma unroll
    for (int hf = 0; hf < D / 128; ++hf) {
      const float4 v = ld_cg_f4(row + 128 * hf + 4 * lane);
      x[(4 * hf) % (D / 32)] = v.x;
      x[(4 * hf + 1) % (D / 32)] = v.y;
      x[(4 * hf + 2) % (D / 32)] = v.z;
      x[(4 * hf + 3) % (D / 32)] = v.w;
    }
  }
}
template <int D>
__device__ __forceinline__ void st_row(float* row, int lane, const float (&x)[D / 32]) {
  if (D == 64) {
    *reinterpret_cast<float2*>(row + 2 * lane) = make_float2(x[0], x[D / 32 - 1]);
  } else {
#pragma unroll
    for (int hf = 0; hf < D / 128; ++hf)
      *reinterpret_cast<float4*>(row + 128 * hf + 4 * lane) =
          make_float4(x[(4 * hf) % (D / 32)], x[(4 * hf + 1) % (D / 32)], x[(4 * hf + 2) % (D / 32)],
                      x[(4 * hf + 3) % (D / 32)]);
  }
}

__device__ __forceinline__ float2 half2_to_float2(uint32_t a) {
  return __half22float2(*reinterpret_cast<const __half2*>(&a));
}

// 8x8 transpose of 16-bit elements across the warp (C-fragment rows -> B-fragment columns).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}


__device__ __forceinline__ void seq_packed(const LayerView& lv, int slot, int& L, int& Np, int& P) {
  L = lv.state[2 * slot];
  const int F = lv.state[2 * slot + 1];
  Np = L > 0 ? kPage * ((L - 1) / kPage) : 0;
  P = Np + F;
}

// Cache slot of (virtual) row b, and the number of the sequence's tokens it attends to: all L for
// decode; for query i of a prefill chunk of n_q queries (the sequence's last n_q tokens) the first
// L - (n_q - 1 - i), i.e. every position up to its own (causal); 0 for padding rows (i >= n_q).
__device__ __forceinline__ int row_slot(const DecodeArgs& a, int b) { return a.seq_ids[a.qpr > 1 ? b / a.qpr : b]; }
__device__ __forceinline__ int row_len(const DecodeArgs& a, int b, int L) {
  if (a.qpr <= 1) return L;
  const int i = b % a.qpr, nq = a.n_q[b / a.qpr];
  return i < nq ? max(0, L - (nq - 1 - i)) : 0;
}

template <int D>
__host__ __device__ constexpr int decode_threads();
// Floats of the d=256 partial-score exchange buffer of a split CTA ([NT][2 tiles][8]).
template <int D>
__host__ __device__ constexpr int decode_xbuf_floats() {
  return D == 256 ? decode_threads<D>() * 2 * 8 : 0;
}

// Split CTAs run `decode_streams` independent page streams of 4 token-group warps x (d/128) coordinate
// halves: 3 streams (12 warps, one CTA per SM) for head_dim 128, 1 stream (8 warps) for head_dim 256.
// (Four streams of 16 warps measured slower at batch 1 and no faster at batch 32.)
template <int D>
__host__ __device__ constexpr int decode_streams() {
  return D <= 128 ? 3 : 1;
}
// Coordinates of one warp (a 128-coordinate half, or all 64) and key-MMA k-steps per warp.
template <int D>
__host__ __device__ constexpr int warp_coords() {
  return D < 128 ? D : 128;
}
template <int D>
__host__ __device__ constexpr int decode_threads() {
  return decode_streams<D>() * 32 * 4 * (D / warp_coords<D>());
}

// =============================================================================================
// Query prep: q_rot = Pi q, q_proj = S q_rot; f16 operands of the three key bit-plane MMAs
// =============================================================================================

// B-operand planes of the key MMAs:
//   key_bits 3: index planes 0, 1 and the QJL sign plane 2; at head_dim 64 and 128 also plane 3, the f16
//     rounding remainder of plane 0's operand, multiplied against plane 0's bits. The f16 rounding of
//     the query operands is the largest error of the estimate; the remainder roughly halves it (at
//     head_dim 128 it took an early prefill query over 1025 tokens with x10 key outliers from 2.6e-3 to
//     inside the 2e-3 attention bound).
//   key_bits 4: index planes 0-3 (3 = parity plane), the QJL sign plane 4, and plane 5, the remainder
//     of plane 0 (the largest weight). Without it the f16 rounding of four index operands adds about
//     1.2x the score error of the 2-bit index.
__host__ __device__ constexpr int key_bplanes(int kb, int d) { return kb == 3 ? (d <= 128 ? 4 : 3) : 6; }
// B plane that carries the QJL operand, and the remainder plane of plane 0 (-1: none).
__host__ __device__ constexpr int key_qjl_plane(int kb) { return kb == 3 ? 2 : 4; }
__host__ __device__ constexpr int key_rem_plane(int kb, int d) { return kb == 3 ? (d <= 128 ? 3 : -1) : 5; }

// Query columns of a split CTA: the 8 B columns of the MMAs carry the kMaxG heads of QP query rows
// (QP = 1 for decode; 2 for prefill, whose chunk queries of one sequence share the key operands).
template <int QP>
__host__ __device__ constexpr int qcols() {
  return kMaxG * QP;
}

// Bytes of a split CTA's query-prep scratch.
template <int D, int KB, int QP = 1>
__host__ __device__ constexpr size_t prep_scratch_bytes() {
  // q_rot, q_proj [columns][D] fp32; 32 floats of scales; B fragments [planes D/16 items][32 lanes]
  // uint2; per-warp offset sums [warps][2 columns]
  return sizeof(float) * (2 * qcols<QP>() * D + 32) + 8 * 32 * (key_bplanes(KB, D) * D / 16) +
         sizeof(float) * 2 * qcols<QP>() * (decode_threads<D>() / 32);
}

// 2^(24 - pos) for the f16 bit position that carries coordinate pair q = 2s + sub (kpair_pos).
__host__ __device__ constexpr float key_prescale(int q) { return (float)(1u << (24 - (q < 12 ? q : q - 4))); }

// Query prep of one (row, KV head), run by every split CTA of that unit (all NT threads):
//   q_rot = Pi q (warp-per-head FWHT), q_proj = S q_rot (m16n8k16 with A = S in f16 from the tables
//   and B = q_rot split into f16 hi + lo), then the f16 B fragments of the three key bit-plane MMAs
//   for this warp's coordinate half and the per-head constants of the score epilogue.
// The B operand of plane pi at coordinate j is w_pi * lambda * x_j * 2^(24 - pos(j)), with w = 2 alpha,
// 2 beta (x = q_rot) or 2 (x = q_proj) and lambda a power of two that puts the largest operand in
// [2^14, 2^15). um / uq undo lambda (and apply the softmax scale in log2 units); cm / cq are half the
// sums of the represented (rounded) operands, i.e. the +-1 offsets of the bit planes.
// A fragments of S (f16) that this warp's q_proj rows need: m-tiles 2 warp + {0, 1}. For head_dim 128
// they are loaded into registers before the kernel waits on earlier stream work (the tables are
// constant); for head_dim 256 query_prep loads them itself.
template <int D>
struct SFrag {
  uint4 a[D == 128 ? 2 : 1][D == 128 ? D / 16 : 1];
};
template <int D>
__device__ __forceinline__ void sfrag_prefetch(const LayerView& lv, SFrag<D>& f) {
  if (D == 128 && (threadIdx.x >> 5) < D / 32) {  // warps that compute q_proj rows
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int m2 = 0; m2 < 2; ++m2)
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) f.a[m2 % (D == 128 ? 2 : 1)][ks % (D == 128 ? D / 16 : 1)] =
          lv.S_frag[sfrag_idx(D, 2 * warp + m2, ks, lane)];
  }
}

// Query prep of one (row, KV head), run by every split CTA of that unit (all NT threads):
//   q_rot = Pi q (warp-per-head FWHT), q_proj = S q_rot (m16n8k16 with A = S in f16 from the tables
//   and B = q_rot split into f16 hi + lo), then the f16 B fragments of the three key bit-plane MMAs
//   for this warp's coordinate half and the per-head constants of the score epilogue.
// The B operand of plane pi at coordinate j is w_pi * lambda * x_j * 2^(24 - pos(j)), with w = 2 alpha,
// 2 beta (x = q_rot) or 2 (x = q_proj). lambda is a power of two that keeps every operand below 2^15
// (f16 max 65504), from bounds: max|w x_j| 2^24 with max|q_proj| <= max_i sum_j |S_ij| * max|q_rot|.
// um / uq undo lambda (and apply the softmax scale in log2 units); cm / cq are half the sums of the
// represented (rounded) operands, i.e. the +-1 offsets of the bit planes.
// With QP = 2 the CTA's row b covers the query rows 2b and 2b + 1 of one sequence: B column n is head
// n % 4 of query n / 4.
template <int D, int NT, int KB, int QP = 1>
__device__ __forceinline__ void query_prep(const DecodeArgs& a, int b, int h, float* ps, const SFrag<D>& sf,
                                           float (&um)[2], float (&cm)[2], float (&uq)[2], float (&cq)[2]) {
  constexpr int NCOL = qcols<QP>();
  constexpr int NBP = key_bplanes(KB, D), QJP = key_qjl_plane(KB), RP = key_rem_plane(KB, D);
  constexpr int NMW = KB == 3 ? 2 : 4;  // index-plane weights
  constexpr int NE = D / 32;
  constexpr int HALVES = D / warp_coords<D>();
  constexpr int MT = D / 16;
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int G = lv.G;
  float wmax = 0.f;  // largest |2 w| of the index planes
#pragma unroll
  for (int p = 0; p < NMW; ++p) wmax = fmaxf(wmax, fabsf(2.f * lv.cb[kCbW + p]));
  float* qr = ps;              // [NCOL][D]
  float* qp = qr + NCOL * D;   // [NCOL][D]
  float* red = qp + NCOL * D;  // [col]: projection lambda; [NCOL + 2 col + {0, 1}]: operand lambdas
  if (warp < NCOL) {           // q_rot: warp w rotates column w (zero rows for heads >= G)
    const int hw = warp % kMaxG, vrow = QP * b + warp / kMaxG;
    float x[NE];
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const int j = lane_coord<D>(e, lane);
      const float qv = hw < G ? bf16_to_f32(a.q[((size_t)vrow * lv.Hq + h * G + hw) * D + j]) : 0.f;
      x[e] = qv * lv.D[j];
    }
    warp_fwht<NE>(x, lane);
    const float rs = rsqrtf((float)D);
    float mx = 0.f;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const float v = x[e] * rs;
      qr[warp * D + lane_coord<D>(e, lane)] = v;
      mx = fmaxf(mx, fabsf(v));
    }
    mx = warp_max(mx);
    if (lane == 0) {
      const float big = 16777216.f;  // 2^24, the largest bit-plane prescale
      red[warp] = mx > 0.f ? exp2f(floorf(log2f(16384.f / mx))) : 1.f;
      const float bm = wmax * mx * big, bp = 2.f * lv.cb[kCbSmax] * mx * big;
      red[NCOL + 2 * warp + 0] = bm > 0.f ? exp2f(floorf(log2f(32768.f / bm))) : 1.f;
      red[NCOL + 2 * warp + 1] = bp > 0.f ? exp2f(floorf(log2f(32768.f / bp))) : 1.f;
    }
  }
  __syncthreads();
  if (warp < MT / 2) {  // q_proj rows 16 mt .. 16 mt + 15, mt = 2 warp + {0, 1}; B column n = column g (zero for g >= NCOL)
    const bool col = g < NCOL;
    const float lam = col ? red[g] : 0.f;
    const float* qrow = qr + (col ? g : 0) * D + 2 * c;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < MT; ++ks) {
      const float x0 = qrow[16 * ks] * lam, x1 = qrow[16 * ks + 1] * lam;
      const float x2 = qrow[16 * ks + 8] * lam, x3 = qrow[16 * ks + 9] * lam;
      const uint32_t h0 = pack_half2(x0, x1), h1 = pack_half2(x2, x3);
      const float2 r0 = half2_to_float2(h0), r1 = half2_to_float2(h1);
      const uint32_t l0 = pack_half2(x0 - r0.x, x1 - r0.y), l1 = pack_half2(x2 - r1.x, x3 - r1.y);
#pragma unroll
      for (int m2 = 0; m2 < 2; ++m2) {
        const uint4 A = D == 128 ? sf.a[m2 % (D == 128 ? 2 : 1)][ks % (D == 128 ? MT : 1)]
                                 : lv.S_frag[sfrag_idx(D, 2 * warp + m2, ks, lane)];
        mma_f16(acc[m2], A.x, A.y, A.z, A.w, h0, h1);
        mma_f16(acc[m2], A.x, A.y, A.z, A.w, l0, l1);
      }
    }
    if (2 * c < NCOL) {  // C columns 2c, 2c + 1 are query columns
      const float i0 = 1.f / red[2 * c], i1 = 1.f / red[2 * c + 1];
#pragma unroll
      for (int m2 = 0; m2 < 2; ++m2) {
        const int r = 16 * (2 * warp + m2) + g;
        qp[(2 * c) * D + r] = acc[m2][0] * i0;
        qp[(2 * c + 1) * D + r] = acc[m2][1] * i1;
        qp[(2 * c) * D + r + 8] = acc[m2][2] * i0;
        qp[(2 * c + 1) * D + r + 8] = acc[m2][3] * i1;
      }
    }
  }
  __syncthreads();
  // B fragments: item (hv, pi, s) is computed by warp item % NW and shared through shared memory;
  // wsum[w][hd] / wsum[w][4 + hd] hold warp w's offset sums of head hd, added in a fixed order below
  // (the same constants in every split CTA and every call)
  constexpr int KS = warp_coords<D>() / 16;  // key-MMA k-steps per warp
  constexpr int NW = NT / 32, NITEMS = HALVES * NBP * KS;
  uint2* frag = reinterpret_cast<uint2*>(red + 32);  // [NITEMS][32]
  float* wsum = reinterpret_cast<float*>(frag + NITEMS * 32);  // [NW][2 NCOL]
  const bool live = g < NCOL && g % kMaxG < G;
  const float lam_m = live ? red[NCOL + 2 * g] : 0.f, lam_q = live ? red[NCOL + 2 * g + 1] : 0.f;
  const float* bm = qr + (live ? g : 0) * D;
  const float* bp = qp + (live ? g : 0) * D;
  __syncthreads();
  float sum_m = 0.f, sum_q = 0.f;
  for (int item = warp; item < NITEMS; item += NW) {
    const int s = item % KS, pi = (item / KS) % NBP, hv = item / (NBP * KS);
    const bool qjl = pi == QJP, rem = pi == RP;  // rem: remainder plane of plane 0
    const float w = qjl ? 2.f * lam_q : 2.f * lv.cb[kCbW + (rem ? 0 : pi)] * lam_m;
    const float* base = qjl ? bp : bm;
    const int j0 = 128 * hv + 16 * s + 2 * c, j1 = j0 + 8;
    const float pre0 = key_prescale(2 * s), pre1 = key_prescale(2 * s + 1);
    const float2 x0 = *reinterpret_cast<const float2*>(base + j0);
    const float2 x1 = *reinterpret_cast<const float2*>(base + j1);
    float v4[4] = {w * x0.x * pre0, w * x0.y * pre0, w * x1.x * pre1, w * x1.y * pre1};
    if (rem) {  // what the f16 operand of plane 0 left out
      const float2 h0 = half2_to_float2(pack_half2(v4[0], v4[1])), h1 = half2_to_float2(pack_half2(v4[2], v4[3]));
      v4[0] -= h0.x;
      v4[1] -= h0.y;
      v4[2] -= h1.x;
      v4[3] -= h1.y;
    }
    const uint32_t b0 = pack_half2(v4[0], v4[1]);
    const uint32_t b1 = pack_half2(v4[2], v4[3]);
    frag[item * 32 + lane] = make_uint2(b0, b1);
    const float2 r0 = half2_to_float2(b0), r1 = half2_to_float2(b1);
    const float v = (r0.x + r0.y) * (1.f / pre0) + (r1.x + r1.y) * (1.f / pre1);
    if (qjl) sum_q += v;
    else sum_m += v;
  }
  sum_m += __shfl_xor_sync(0xffffffffu, sum_m, 1);
  sum_m += __shfl_xor_sync(0xffffffffu, sum_m, 2);
  sum_q += __shfl_xor_sync(0xffffffffu, sum_q, 1);
  sum_q += __shfl_xor_sync(0xffffffffu, sum_q, 2);
  if (c == 0 && g < NCOL) {
    wsum[warp * 2 * NCOL + g] = sum_m;
    wsum[warp * 2 * NCOL + NCOL + g] = sum_q;
  }
  __syncthreads();
  const float kappa = 1.2533141373155003f / (float)D;  // sqrt(pi/2) / d
#pragma unroll
  for (int i = 0; i < 2; ++i) {  // C-fragment column 2c + i is query column hd
    const int hd = min(2 * c + i, NCOL - 1);
    float sm = 0.f, sq = 0.f;
    for (int w = 0; w < NW; ++w) {
      sm += wsum[w * 2 * NCOL + hd];
      sq += wsum[w * 2 * NCOL + NCOL + hd];
    }
    um[i] = a.scale * kLog2e / red[NCOL + 2 * hd];
    cm[i] = 0.5f * sm;
    uq[i] = a.scale * kLog2e * kappa / red[NCOL + 2 * hd + 1];
    cq[i] = 0.5f * sq;
  }
}

// =============================================================================================
// Split-K decode over packed pages (blockIdx.x < n_splits) and the exact ring split (== n_splits)
// =============================================================================================
// Ring split shared memory: K rows (and, for head_dim 128, V rows next to them, so both copies are
// in flight together), then [128][4] scores, the softmax statistics and q as fp32 [4][D].
template <int D>
__host__ __device__ constexpr bool ring_kv_together() {
  return D <= 128;
}
template <int D, int QP = 1>
__host__ __device__ constexpr size_t ring_smem_bytes() {
  return 128 + (ring_kv_together<D>() ? 2 : 1) * 2 * kPage * D + kPage * qcols<QP>() * 4 + 16 * qcols<QP>() +
         qcols<QP>() * D * 4;
}

// A partial of `ncol` query columns: m [ncol], l [ncol], o [ncol][D].
__device__ __forceinline__ void write_empty_partial(float* part, int D, int tid, int nt, int ncol = kMaxG) {
  for (int i = tid; i < 2 * ncol + ncol * D; i += nt) part[i] = i < ncol ? -INFINITY : 0.f;
}

// Exact attention over the unflushed ring tokens [F, R) of one (row, KV head). K and V rows are
// bulk-copied into shared memory (together for head_dim 128). Scores are thread-per-token: thread t
// walks its K row in 16-byte chunks starting at chunk t, so the 8 lanes of each quarter-warp read
// 8 different bank groups. P.V is thread-per-coordinate.
// With QP = 2 the CTA's query rows 2b, 2b + 1 see n0 and n1 ring tokens (causal; a padding row sees
// none): the columns of each query take no weight from ring tokens past its own count.
// Returns false when a copy into shared memory may still be in flight (a wait gave up and so did the
// bounded drain after it): the CTA must then not reuse its shared memory.
template <int D, int NT, int QP = 1>
__device__ __noinline__ bool ring_split(const DecodeArgs& a, int b, int h, int slot, float* part, uint8_t* smem_raw) {
  constexpr int NC = D / 8;  // 16-byte chunks per row
  constexpr int NCOL = qcols<QP>();
  constexpr bool KV = ring_kv_together<D>();
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int L, Np, P;
  seq_packed(lv, slot, L, Np, P);
  // ring tokens are positions P .. Lq - 1 of each query row
  const int n0 = row_len(a, QP * b, L) - P, n1 = QP == 1 ? n0 : row_len(a, QP * b + 1, L) - P;
  const int F = P - Np, n = max(n0, n1);
  if (n <= 0) {
    write_empty_partial(part, D, tid, NT, NCOL);
    return true;
  }
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw);
  const uint16_t* krows = reinterpret_cast<const uint16_t*>(smem_raw + 128);  // [n][D] bf16
  const uint16_t* vrows = KV ? krows + (size_t)kPage * D : krows;             // [n][D] bf16
  float* sc = reinterpret_cast<float*>(smem_raw + 128 + (KV ? 2 : 1) * 2 * kPage * D);  // [128][NCOL]
  float* red = sc + kPage * NCOL;                                                        // [NCOL][2] (+ pad)
  float* qs = red + 4 * NCOL;                                                            // [NCOL][D]
  const uint16_t* rk = lv.ring + (((size_t)slot * lv.Hkv + h) * 2) * kPage * D + (size_t)F * D;
  const uint16_t* rv = rk + (size_t)kPage * D;
  const uint32_t bytes = (uint32_t)n * D * 2;
  if (tid == 0) {
    mbar_init(bar, 1);
    if (KV) mbar_init(bar + 1, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    mbar_expect_tx(bar, bytes);
    bulk_g2s(smem_raw + 128, rk, bytes, bar);
    if (KV) {
      mbar_expect_tx(bar + 1, bytes);
      bulk_g2s(smem_raw + 128 + 2 * kPage * D, rv, bytes, bar + 1);
    }
  }
  const int G = lv.G;
  for (int i = tid; i < NCOL * D; i += NT) {
    const int g = (i / D) % kMaxG, vrow = QP * b + i / (kMaxG * D);
    qs[i] = g < G ? bf16_to_f32(a.q[((size_t)vrow * lv.Hq + h * G + g) * D + (i % D)]) : 0.f;
  }
  // every thread agrees on whether the K rows landed (the V copy below depends on it)
  const bool ok_k = __syncthreads_and(mbar_wait(bar, 0)) != 0;
  const float s2 = a.scale * kLog2e;
  if (ok_k) {
    for (int t = tid; t < n; t += NT) {
      float acc[NCOL];
#pragma unroll
      for (int g = 0; g < NCOL; ++g) acc[g] = 0.f;
      const uint16_t* row = krows + (size_t)t * D;
#pragma unroll 4
      for (int i = 0; i < NC; ++i) {
        const int ci = (i + t) & (NC - 1);
        const uint4 u = *reinterpret_cast<const uint4*>(row + 8 * ci);
        const float k[8] = {__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                            __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u),
                            __uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u),
                            __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u)};
#pragma unroll
        for (int g = 0; g < NCOL; ++g) {
          const float4 q0 = *reinterpret_cast<const float4*>(qs + g * D + 8 * ci);
          const float4 q1 = *reinterpret_cast<const float4*>(qs + g * D + 8 * ci + 4);
          acc[g] = fmaf(q0.x, k[0], fmaf(q0.y, k[1], fmaf(q0.z, k[2], fmaf(q0.w, k[3], acc[g]))));
          acc[g] = fmaf(q1.x, k[4], fmaf(q1.y, k[5], fmaf(q1.z, k[6], fmaf(q1.w, k[7], acc[g]))));
        }
      }
#pragma unroll
      for (int g4 = 0; g4 < NCOL; g4 += 4)
        *reinterpret_cast<float4*>(sc + t * NCOL + g4) =
            make_float4(acc[g4] * s2, acc[g4 + 1] * s2, acc[g4 + 2] * s2, acc[g4 + 3] * s2);
    }
  }
  __syncthreads();  // every K row has been read
  if (!KV && tid == 0 && ok_k) {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    mbar_expect_tx(bar, bytes);
    bulk_g2s(smem_raw + 128, rv, bytes, bar);
  }
  if (warp < NCOL) {  // softmax statistics: warp g reduces column g over its query's ring tokens
    const int nw = warp < kMaxG ? n0 : n1;
    float m = -INFINITY;
    for (int t = lane; t < nw; t += 32) m = fmaxf(m, sc[t * NCOL + warp]);
    m = warp_max(m);
    float l = 0.f;
    for (int t = lane; t < nw; t += 32) {
      const float p = exp2f(sc[t * NCOL + warp] - m);
      sc[t * NCOL + warp] = p;
      l += p;
    }
    for (int t = max(nw, 0) + lane; t < n; t += 32) sc[t * NCOL + warp] = 0.f;  // past this query's position
    l = warp_sum(l);
    if (lane == 0) {
      red[2 * warp] = m;
      red[2 * warp + 1] = l;
    }
  }
  __syncthreads();
  const bool ok_v = __syncthreads_and(ok_k && mbar_wait(KV ? bar + 1 : bar, KV ? 0 : 1)) != 0;
  if (!ok_v) {
    // a wait gave up: thread 0 waits (bounded) for the copies that were issued and not seen to land -
    // K (if its wait failed) and V (issued with K, or after K landed) - so that none lands later
    bool drained = true;
    if (tid == 0) {
      set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
      if (!ok_k) drained = mbar_wait(bar, 0);
      if (KV) drained = mbar_wait(bar + 1, 0) && drained;
      else if (ok_k) drained = mbar_wait(bar, 1) && drained;
    }
    write_empty_partial(part, D, tid, NT, NCOL);
    return __syncthreads_and(drained) != 0;
  }
  for (int j = tid; j < D; j += NT) {
    float o[2][NCOL];
#pragma unroll
    for (int g = 0; g < NCOL; ++g) o[0][g] = o[1][g] = 0.f;
    int t = 0;
#pragma unroll 4
    for (; t + 1 < n; t += 2) {  // two independent accumulator sets
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float vv = bf16_to_f32(vrows[(size_t)(t + u) * D + j]);
#pragma unroll
        for (int g4 = 0; g4 < NCOL; g4 += 4) {
          const float4 p = *reinterpret_cast<const float4*>(sc + (t + u) * NCOL + g4);
          o[u][g4] = fmaf(p.x, vv, o[u][g4]);
          o[u][g4 + 1] = fmaf(p.y, vv, o[u][g4 + 1]);
          o[u][g4 + 2] = fmaf(p.z, vv, o[u][g4 + 2]);
          o[u][g4 + 3] = fmaf(p.w, vv, o[u][g4 + 3]);
        }
      }
    }
    if (t < n) {
      const float vv = bf16_to_f32(vrows[(size_t)t * D + j]);
#pragma unroll
      for (int g4 = 0; g4 < NCOL; g4 += 4) {
        const float4 p = *reinterpret_cast<const float4*>(sc + t * NCOL + g4);
        o[0][g4] = fmaf(p.x, vv, o[0][g4]);
        o[0][g4 + 1] = fmaf(p.y, vv, o[0][g4 + 1]);
        o[0][g4 + 2] = fmaf(p.z, vv, o[0][g4 + 2]);
        o[0][g4 + 3] = fmaf(p.w, vv, o[0][g4 + 3]);
      }
    }
#pragma unroll
    for (int g = 0; g < NCOL; ++g) part[2 * NCOL + g * D + j] = o[0][g] + o[1][g];
  }
  if (tid < NCOL) {
    part[tid] = red[2 * tid];
    part[NCOL + tid] = red[2 * tid + 1];
  }
  return true;
}

// =============================================================================================
// Combine: LSE merge of history splits (rotated basis) -> Pi^T -> exact merge with the ring split.
// Run by the last CTA of a (row, KV head) to finish its partial. Warp w merges query head w on its
// own (no block barrier): lanes take the splits' (m, l), the weights go through shared memory column w.
// =============================================================================================
template <int D, int NT, int QP = 1>
__device__ __noinline__ void combine_unit(const DecodeArgs& a, int b, int h, float* sm) {
  constexpr int NE = D / 32;
  constexpr int NCOL = qcols<QP>();
  const LayerView& lv = a.lv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp >= NCOL || warp % kMaxG >= lv.G) return;
  const int hd = warp;  // query column (head hd % 4 of query row QP b + hd / 4); lane holds coordinates 4*lane+e (+128)
  const int nsp = a.plan.n_splits;
  const size_t stride = a.plan.part_stride / sizeof(float);
  const float* base = reinterpret_cast<const float*>(a.ws + a.plan.part_off +
                                                     ((size_t)b * lv.Hkv + h) * (nsp + 1) * a.plan.part_stride);
  float* fs = sm;                      // [nsp][NCOL] split maxima, then split weights (column hd is this warp's)
  float* ls = fs + NCOL * (nsp + 1);   // [nsp][NCOL] split sums
  // 0. the outputs of the first PRE splits and the ring partial do not depend on the weights: their
  //    loads share the round trip of the (m, l) loads
  constexpr int PRE = D == 128 ? 20 : D == 64 ? 24 : 8;
  const float* ob = base + 2 * NCOL + hd * D;
  const float* rp = base + nsp * stride;
  float vpre[PRE][NE], rvp[NE];
#pragma unroll
  for (int u = 0; u < PRE; ++u) {
    if (u < nsp) {
      ld_cg_row<D>(ob + u * stride, lane, vpre[u]);
    } else {
#pragma unroll
      for (int e = 0; e < NE; ++e) vpre[u][e] = 0.f;
    }
  }
  ld_cg_row<D>(rp + 2 * NCOL + hd * D, lane, rvp);
  const float mr = ld_cg_f(rp + hd), lr = ld_cg_f(rp + NCOL + hd);
  float dsg[NE];  // the rotation signs of this lane's coordinates (constant table)
#pragma unroll
  for (int e = 0; e < NE; ++e) dsg[e] = lv.D[lane_coord<D>(e, lane)];
  // 1. the splits' (m, l) of this head across the lanes; maximum, weights and the weighted sum of l
  float mloc = -INFINITY;
  for (int s = lane; s < nsp; s += 32) {
    const float mv = ld_cg_f(base + s * stride + hd), lv2 = ld_cg_f(base + s * stride + NCOL + hd);
    fs[NCOL * s + hd] = mv;
    ls[NCOL * s + hd] = lv2;
    mloc = fmaxf(mloc, mv);
  }
  const float m = warp_max(mloc);
  float lloc = 0.f;
  for (int s = lane; s < nsp; s += 32) {
    const float mv = fs[NCOL * s + hd];
    const float f = mv == -INFINITY ? 0.f : exp2f(mv - m);
    fs[NCOL * s + hd] = f;
    lloc = fmaf(f, ls[NCOL * s + hd], lloc);
  }
  const float l = warp_sum(lloc);
  __syncwarp();
  // 2. weighted sum of the split outputs: the prefetched PRE, then 16 splits' loads in flight at a time
  float o[NE], o2[NE];
#pragma unroll
  for (int e = 0; e < NE; ++e) o[e] = o2[e] = 0.f;
#pragma unroll
  for (int u = 0; u < PRE; ++u) {
    const float f = u < nsp ? fs[u * NCOL + hd] : 0.f;
    float* acc = (u & 1) ? o2 : o;
#pragma unroll
    for (int e = 0; e < NE; ++e) acc[e] = fmaf(f, vpre[u][e], acc[e]);
  }
  int s0 = PRE;
  for (; s0 + 16 <= nsp; s0 += 16) {  // empty splits hold weight 0 and O = 0
    float v[16][NE];
#pragma unroll
    for (int u = 0; u < 16; ++u) ld_cg_row<D>(ob + (s0 + u) * stride, lane, v[u]);
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float f = fs[(s0 + u) * NCOL + hd];
      float* acc = (u & 1) ? o2 : o;
#pragma unroll
      for (int e = 0; e < NE; ++e) acc[e] = fmaf(f, v[u][e], acc[e]);
    }
  }
  for (; s0 < nsp; ++s0) {
    const float f = fs[s0 * NCOL + hd];
    float v[NE];
    ld_cg_row<D>(ob + s0 * stride, lane, v);
#pragma unroll
    for (int e = 0; e < NE; ++e) o[e] = fmaf(f, v[e], o[e]);
  }
#pragma unroll
  for (int e = 0; e < NE; ++e) o[e] += o2[e];
  // 3. Pi^T o = D * (H o) / sqrt(d), then the exact merge with the ring split
  warp_fwht<NE>(o, lane);
  const float rs = rsqrtf((float)D);
#pragma unroll
  for (int e = 0; e < NE; ++e) o[e] *= rs * dsg[e];
  const float mm = fmaxf(m, mr);
  const float fh = (m == -INFINITY) ? 0.f : exp2f(m - mm);
  const float fr = (mr == -INFINITY) ? 0.f : exp2f(mr - mm);
  const float den = fh * l + fr * lr;
  const float inv = den > 0.f ? 1.f / den : 0.f;
  float r[NE];
#pragma unroll
  for (int e = 0; e < NE; ++e) r[e] = (fh * o[e] + fr * rvp[e]) * inv;
  st_row<D>(a.out + ((size_t)(QP * b + hd / kMaxG) * lv.Hq + h * lv.G + hd % kMaxG) * D, lane, r);
}

// Zero outputs of the query columns of (row b, KV head h): the result of a unit whose last CTA cannot
// use its shared memory (a copy into it may still be in flight after a wait gave up; the call has
// TQ_DEV_ERR_TIMEOUT set and its result is unspecified).
template <int D, int NT, int QP>
__device__ __forceinline__ void zero_unit_out(const DecodeArgs& a, int b, int h) {
  constexpr int NCOL = qcols<QP>();
  const LayerView& lv = a.lv;
  for (int i = threadIdx.x; i < NCOL * D; i += NT) {
    const int col = i / D;
    if (col % kMaxG < lv.G)
      a.out[((size_t)(QP * b + col / kMaxG) * lv.Hq + h * lv.G + col % kMaxG) * D + i % D] = 0.f;
  }
}

// After this CTA's partial is written: the last of the (n_splits + 1) CTAs of the (row, KV head)
// merges all of them (an arrival counter; no CTA waits on another). smem_ok = false: this CTA's shared
// memory may still receive a copy, so a last CTA writes zeros instead of combining.
template <int D, int NT, int QP = 1>
__device__ __noinline__ void finish_unit(const DecodeArgs& a, int b, int h, uint8_t* smem, bool smem_ok = true) {
  __shared__ int s_last;
  __syncthreads();  // every thread's part of the partial is written
  if (threadIdx.x == 0) {
    // acq_rel at gpu scope: releases this CTA's partial (ordered before by the barrier) and, in the
    // last CTA, acquires every other CTA's
    int* cnt = reinterpret_cast<int*>(a.ws + a.plan.cnt_off) + b * a.lv.Hkv + h;
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;\n" : "=r"(old) : "l"(cnt) : "memory");
    s_last = old == a.plan.n_splits;
    if (s_last) *cnt = 0;  // ready for the next call
  }
  __syncthreads();
  if (!s_last) return;
  if (!smem_ok) {
    zero_unit_out<D, NT, QP>(a, b, h);
    return;
  }
  combine_unit<D, NT, QP>(a, b, h, reinterpret_cast<float*>(smem + 128));
}

// Split-K decode CTA: 4 token groups x (d/128) coordinate halves of warps. Warp (tg, hf) owns
// tokens 32tg..32tg+31 of every page and coordinates 128hf..128hf+127.
// Scores: each 16-token tile is three bit-plane m16n8k16 MMA chains. A = masked key bits
// (f16 2^(q-24) or 0), B = prepped f16 query (4 heads + 4 zero columns). For d=256 the two halves
// exchange partial sums through shared memory.
// Values: P is moved from C to B fragment layout with movmatrix and scaled per value group. Then
// P.V runs on m16n8k16 with A = code fields (f16 subnormals code * 2^(pos-24)).
// QP = 2 (prefill): the CTA's row b is the query rows 2b and 2b + 1 of one sequence, in the 8 B
// columns; each lane's two C columns belong to query c / 2.
// head_dim 256 with 2-bit values runs two CTAs per SM (128 registers, 104 KB of shared memory each);
// its other shapes need more than half of an SM's shared memory and keep one.
template <int D, int VB, int STAGES, bool PAGED, int KB, int QP = 1>
__global__ void __launch_bounds__(decode_threads<D>(), D == 256 && VB == 2 ? 2 : 1) k_decode(DecodeArgs a) {
  constexpr int NCOL = qcols<QP>();
  constexpr int NBP = key_bplanes(KB, D);  // B planes of the key MMAs (stored planes: KB)
  constexpr int RP = key_rem_plane(KB, D);
  constexpr int CW = warp_coords<D>();  // coordinates per warp
  constexpr int HALVES = D / CW;
  constexpr int KS = CW / 16;           // key-MMA k-steps per warp
  constexpr int QG = CW / 32;           // value groups per warp
  constexpr int NT = decode_threads<D>();
  constexpr int NS = decode_streams<D>();
  constexpr int SW = 4 * HALVES;  // warps per stream
  constexpr int NG = D / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const LayerView& lv = a.lv;
  const int sp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int stream = warp / SW, tg = warp & 3, hf = (warp % SW) >> 2;
  const int nsp = a.plan.n_splits;
  float* part = reinterpret_cast<float*>(a.ws + a.plan.part_off +
                                         (((size_t)b * lv.Hkv + h) * (nsp + 1) + sp) * a.plan.part_stride);
  // Every kernel of this library starts its dependents only after its own stream wait, so what this
  // kernel reads before its wait (q, seq_ids, the tables, the packed pages and count) was complete
  // before the previous kernel's dependents started.
  const int slot = row_slot(a, QP * b);
  // The sequence state is read below before the stream wait. A decode row's packed count does not
  // depend on the length that an append which codes no page may still be writing (such an append
  // releases its dependents early). A prefill query's causal length does; a prefill launch never
  // overlaps an append, because tq_prefill_attention zeroes the arrival counters with a memset right
  // before this kernel, and a memset waits for the whole preceding kernel.
  if (slot < 0 || slot >= lv.max_seqs) {
    pdl_wait();
    pdl_launch();
    write_empty_partial(part, D, tid, NT, NCOL);
    finish_unit<D, NT, QP>(a, b, h, smem);
    return;
  }
  if (sp == nsp) {
    pdl_wait();
    pdl_launch();
    const bool smem_ok = ring_split<D, NT, QP>(a, b, h, slot, part, smem);
    finish_unit<D, NT, QP>(a, b, h, smem, smem_ok);
    return;
  }
  int L, Np, P;
  seq_packed(lv, slot, L, Np, P);
  // a prefill query sees the packed tokens before its own position; Pq: this lane's query
  const int P0 = min(P, row_len(a, QP * b, L)), P1 = QP == 1 ? P0 : min(P, row_len(a, QP * b + 1, L));
  const int Pq = (QP == 1 || (lane & 3) < 2) ? P0 : P1;
  P = max(P0, P1);
  const int n_pages = (P + kPage - 1) / kPage;
  const int pps = a.plan.pages_per_split;
  if (sp == 0 && tid == 0 && n_pages > nsp * pps) set_status(lv.status, TQ_DEV_ERR_SPLITS);
  const int pg0 = sp * pps, pg1 = min(n_pages, pg0 + pps);
  if (pg0 >= pg1) {
    pdl_wait();
    pdl_launch();
    write_empty_partial(part, D, tid, NT, NCOL);
    finish_unit<D, NT, QP>(a, b, h, smem);
    return;
  }
  const PageLayout pl = page_layout(D, VB, KB);
  const uint32_t PB = pl.bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [stream][stage]
  uint8_t* stage0 = smem + 128;                         // [stream][stage] pages
  float* xbuf = reinterpret_cast<float*>(stage0 + (size_t)NS * STAGES * PB);  // [NT][2 tiles][8] partial scores
  // contiguous cache: the pages of (slot, h) follow each other; a paged cache maps every page through the
  // block table (a separate instantiation: the lookup inside the page loop costs the contiguous kernel
  // about 20 % if it is only branched around)
  const uint8_t* gpages = lv.pages + ((size_t)slot * lv.Hkv + h) * lv.max_pages * PB;
  const int npg = pg1 - pg0;  // stream st takes local pages st, st + NS, st + 2 NS, ...
  // wait-timeout test hook (head_dim 128 kernels): this CTA's stream 0 gets no copy (and no expect_tx) for
  // page stage fault_k
  const int fault_k =
      (D == 128 && a.fault_stage >= 0 && a.fault_stage < STAGES && sp == 0 && h == 0 && b == 0) ? a.fault_stage : -1;
  if (tid == 0) {
    for (int s = 0; s < NS * STAGES; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    for (int st = 0; st < NS; ++st)
      for (int s = 0; s < STAGES && st + NS * s < npg; ++s) {
        if (st == 0 && s == fault_k) continue;
        if (PAGED) {  // a page without a block reads block 0 and is reported after the loop
          const int blk = lv.btab[(size_t)slot * lv.max_pages + pg0 + st + NS * s];
          const bool okb = (unsigned)blk < (unsigned)lv.n_blocks;
          if (!okb) set_status(lv.status, TQ_DEV_ERR_BLOCK);
          mbar_expect_tx(&full[st * STAGES + s], PB);
          bulk_g2s(stage0 + (size_t)(st * STAGES + s) * PB, lv.pages + ((size_t)(okb ? blk : 0) * lv.Hkv + h) * PB, PB,
                   &full[st * STAGES + s]);
        } else {
          mbar_expect_tx(&full[st * STAGES + s], PB);
          bulk_g2s(stage0 + (size_t)(st * STAGES + s) * PB, gpages + (size_t)(pg0 + st + NS * s) * PB, PB,
                   &full[st * STAGES + s]);
        }
      }
  }
  SFrag<D> sfrag;
  sfrag_prefetch<D>(lv, sfrag);
  float um[2], cm[2], uq[2], cq[2];
  float* ps = xbuf + decode_xbuf_floats<D>();
  query_prep<D, NT, KB, QP>(a, b, h, ps, sfrag, um, cm, uq, cq);  // shared memory only
  pdl_wait();  // the partials and counters of any decode that shares ws are no longer in use
  pdl_launch();
  // f16 B fragments of the key MMAs for this warp's coordinate half, [plane][k-step][lane] in shared
  // memory (written by query_prep; read once per page and k-step, shared by both tiles)
  const uint2* bfr = reinterpret_cast<const uint2*>(ps + 2 * NCOL * D + 32) + hf * NBP * KS * 32 + lane;
  const int g = lane >> 2, c = lane & 3;
  // score = n (um (am - cm) + uq gamma (aq - cq)) as n fma(gamma, fma(uq, aq, -uq cq), fma(um, am, -um cm)).
  // Columns of heads >= G (and, for decode, columns 4..7) carry zero query operands: their scores are
  // finite and their outputs are never merged, so only tokens past the end of the tokens this lane's
  // query sees need masking (a partial last page, or a prefill query's causal end).
  float umcm[2], uqcq[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    umcm[i] = um[i] * cm[i];
    uqcq[i] = uq[i] * cq[i];
  }
  float O[2 * QG][4];
#pragma unroll
  for (int mt = 0; mt < 2 * QG; ++mt) O[mt][0] = O[mt][1] = O[mt][2] = O[mt][3] = 0.f;
  float m_eff[2] = {-INFINITY, -INFINITY}, l_acc[2] = {0.f, 0.f};
  __syncthreads();
  // kt: the first page (loop index k) whose wait this thread gave up on, or -1. A wait that gives up
  // marks the call (TQ_DEV_ERR_TIMEOUT); this thread then waits no more, and a stream whose issuing
  // thread gave up issues no more copies. The loop still runs to its end so that every warp reaches the
  // stream barriers (the page contents are then unspecified).
  int kt = -1;
  const bool issuer = (tid % (32 * SW)) == 0;  // the thread that issues this stream's copies
  bool bad_block = false;  // paged cache: a page without a block was read as block 0
  int next_blk = 0;        // paged cache: block of the page this stream's issuing thread copies next
  if (PAGED && issuer && stream + NS * STAGES < npg)
    next_blk = lv.btab[(size_t)slot * lv.max_pages + pg0 + stream + NS * STAGES];

  for (int k = 0; stream + NS * k < npg; ++k) {
    const int ip = stream + NS * k, s_ = k % STAGES;
    if (kt < 0 && !mbar_wait(&full[stream * STAGES + s_], (k / STAGES) & 1,
                             stream == 0 && k == fault_k ? a.fault_polls : kWaitPolls))
      kt = k;
    const uint8_t* pg = stage0 + (size_t)(stream * STAGES + s_) * PB;
    const int valid = min(kPage, Pq - (pg0 + ip) * kPage);  // tokens of this page that this lane's query sees
    const uint2* kw2 = reinterpret_cast<const uint2*>(pg + pl.kbits_off);
    const uint32_t* nrm = reinterpret_cast<const uint32_t*>(pg + pl.norms_off);
    const uint32_t* vsc = reinterpret_cast<const uint32_t*>(pg + pl.vscale_off);  // [token pair][group] f16x2
    float sc[2][4];
    // six independent MMA chains: (tile, chain); both tiles' words are loaded up front. With a 3-bit
    // index the four index planes share two chains (planes 0-1 and 2-3) and the parity plane's
    // words are formed once per page.
    constexpr int NKW = KB == 3 ? 3 : 5;  // key words per tile: the stored planes (+ the parity plane)
    float acc[2][3][4];
    uint2 kwv[2][NKW];
#pragma unroll
    for (int kap = 0; kap < 2; ++kap) {
#pragma unroll
      for (int ch = 0; ch < 3; ++ch) acc[kap][ch][0] = acc[kap][ch][1] = acc[kap][ch][2] = acc[kap][ch][3] = 0.f;
#pragma unroll
      for (int pi = 0; pi < KB; ++pi) {
        uint2 wv;
        if (D == 64) {  // both tiles in one word; the odd tile 8 bit positions higher
          wv = kw2[(tg * KB + pi) * 32 + lane];
          if (kap) wv = make_uint2(wv.x >> 8, wv.y >> 8);
        } else {
          wv = kw2[(((2 * tg + kap) * KB + pi) * HALVES + hf) * 32 + lane];
        }
        kwv[kap][pi == KB - 1 ? NKW - 1 : pi] = wv;  // the sign plane is the last word
      }
      if (KB == 4)
        kwv[kap][3] = make_uint2(kwv[kap][0].x ^ kwv[kap][1].x ^ kwv[kap][2].x, kwv[kap][0].y ^ kwv[kap][1].y ^ kwv[kap][2].y);
    }
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      const int q0 = s < 6 ? 2 * s : 2 * s - 4;
      const uint32_t m0 = 0x00010001u << q0, m1 = 0x00010001u << (q0 + 1);
#pragma unroll
      for (int pi = 0; pi < NBP; ++pi) {
        const uint2 bv = bfr[(pi * KS + s) * 32];
        // chains: key_bits 3 one per plane (the remainder joins plane 0); key_bits 4 {0, 1, 5}, {2, 3}, {4}
        const int ch = KB == 3 ? (pi == RP ? 0 : pi) : (pi == 4 ? 2 : (pi == 2 || pi == 3) ? 1 : 0);
        const int wi = pi == RP ? 0 : pi;  // the remainder plane multiplies plane 0's bits
#pragma unroll
        for (int kap = 0; kap < 2; ++kap) {
          const uint32_t x0 = s < 6 ? kwv[kap][wi].x : kwv[kap][wi].x >> 4;
          const uint32_t x1 = s < 6 ? kwv[kap][wi].y : kwv[kap][wi].y >> 4;
          mma_f16(acc[kap][ch], x0 & m0, x1 & m0, x0 & m1, x1 & m1, bv.x, bv.y);
        }
      }
    }
#pragma unroll
    for (int kap = 0; kap < 2; ++kap) {
      const int tile = 2 * tg + kap;
      float am[4], aq[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        am[i] = acc[kap][0][i] + acc[kap][1][i];
        aq[i] = acc[kap][2][i];
      }
      if (HALVES == 2) {  // add the partner half's partial sums
        float* mine = xbuf + ((size_t)tid * 2 + kap) * 8;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          mine[i] = am[i];
          mine[4 + i] = aq[i];
        }
        named_barrier(1 + tg, 64);
        const float* other = xbuf + ((size_t)(tid ^ 128) * 2 + kap) * 8;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          am[i] += other[i];
          aq[i] += other[4 + i];
        }
      }
      const int t0 = 16 * tile + g, t1 = t0 + 8;
      const uint32_t n0w = nrm[t0], n1w = nrm[t1];
      const float nv[2] = {__half2float(__ushort_as_half((uint16_t)(n0w & 0xffff))),
                           __half2float(__ushort_as_half((uint16_t)(n1w & 0xffff)))};
      const float gv[2] = {__half2float(__ushort_as_half((uint16_t)(n0w >> 16))),
                           __half2float(__ushort_as_half((uint16_t)(n1w >> 16)))};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = i >> 1, col = i & 1;
        sc[kap][i] = nv[row] * fmaf(gv[row], fmaf(uq[col], aq[i], -uqcq[col]), fmaf(um[col], am[i], -umcm[col]));
      }
      if (valid < kPage) {  // the last page of a sequence: tokens past its end take no weight
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (((i >> 1) ? t1 : t0) >= valid) sc[kap][i] = -INFINITY;
      }
    }
    // ---- online softmax (exp2 units); m_eff also keeps p * s * 2^(24 - pos) inside f16 range ----
    float mx[2];
#pragma unroll
    for (int col = 0; col < 2; ++col) {
      float m = fmaxf(fmaxf(sc[0][col], sc[0][2 + col]), fmaxf(sc[1][col], sc[1][2 + col]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
      mx[col] = m;
    }
    // largest value scale of this warp's tokens: the scales are finite non-negative f16, so their bit
    // patterns order like their values (one warp max-reduction on the bits)
    uint32_t smax_bits = 0;
    for (int i = lane; i < 16 * NG; i += 32) smax_bits = __vmaxu2(smax_bits, vsc[16 * tg * NG + i]);
    smax_bits = __reduce_max_sync(0xffffffffu, max(smax_bits & 0xffffu, smax_bits >> 16));
    // e2 = exponent of smax as frexp gives it (biased f16 exponent - 14; <= 0 for subnormals and zero).
    // p * 2^(24-pos) <= 2^(15 - max(e2, 0)) keeps both P (packed before the scale) and P * s below 2^15
    const float E = (float)(9 + max((int)((smax_bits >> 10) & 31u) - 14, 0));
    float alpha[2], m_use[2];  // m_use: m_eff, or 0 while a column has seen no token (then every x is -inf)
#pragma unroll
    for (int col = 0; col < 2; ++col) {
      const float m_new = fmaxf(m_eff[col], mx[col] + E);
      alpha[col] = (m_new == -INFINITY) ? 1.f : exp2f(m_eff[col] - m_new);
      m_eff[col] = m_new;
      m_use[col] = m_new == -INFINITY ? 0.f : m_new;
      l_acc[col] *= alpha[col];
    }
    uint32_t pb[2][2];  // B fragments of P (no value scale yet): [k-step][tokens 0-7 / 8-15]
#pragma unroll
    for (int kap = 0; kap < 2; ++kap) {
      float pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = i >> 1, col = i & 1;
        const float pn = exp2f(sc[kap][i] - m_use[col]);  // exp2(-inf) = 0
        l_acc[col] += pn;
        const int pos = VB == 2 ? vpos2(kap, row) : vpos4(row);
        pv[i] = pn * (float)(1u << (24 - pos));
      }
      pb[kap][0] = movmatrix_trans(pack_half2(pv[0], pv[1]));
      pb[kap][1] = movmatrix_trans(pack_half2(pv[2], pv[3]));
    }
    // ---- P.V, one value group (two m-tiles) of this half at a time ----
    // Each page's product starts from its own mid-rise offset: C = -off * sum_t p_t s_t per head,
    // made by one MMA pair whose A is the constant -(2^VB - 1) * 2^(pos-24) (= -2 off at each token's
    // position) and halved. The codes then add sum_t code_t p_t s_t, so the cancellation between the
    // code sum and the offset stays inside one page, however long the context.
    const uint32_t* vw = reinterpret_cast<const uint32_t*>(pg + pl.vbits_off);
    constexpr uint32_t kVmax = (1u << VB) - 1u;
    constexpr uint32_t kOff00 = voff_pattern(kVmax, VB == 2 ? vpos2(0, 0) : vpos4(0));
    constexpr uint32_t kOff01 = voff_pattern(kVmax, VB == 2 ? vpos2(0, 1) : vpos4(1));
    constexpr uint32_t kOff10 = voff_pattern(kVmax, VB == 2 ? vpos2(1, 0) : vpos4(0));
    constexpr uint32_t kOff11 = voff_pattern(kVmax, VB == 2 ? vpos2(1, 1) : vpos4(1));
#pragma unroll
    for (int q = 0; q < QG; ++q) {
      const int gq = QG * hf + q;
      uint32_t bf[2][2];
#pragma unroll
      for (int kap = 0; kap < 2; ++kap) {
        const int tile = 2 * tg + kap;
        bf[kap][0] = hmul2_u32(pb[kap][0], vsc[(8 * tile + c) * NG + gq]);
        bf[kap][1] = hmul2_u32(pb[kap][1], vsc[(8 * tile + 4 + c) * NG + gq]);
      }
      float coff[4] = {0.f, 0.f, 0.f, 0.f};
      mma_f16(coff, kOff00, kOff00, kOff01, kOff01, bf[0][0], bf[0][1]);
      mma_f16(coff, kOff10, kOff10, kOff11, kOff11, bf[1][0], bf[1][1]);
#pragma unroll
      for (int i = 0; i < 4; ++i) coff[i] *= 0.5f;
#pragma unroll
      for (int mh = 0; mh < 2; ++mh) {
        const int mt = 2 * q + mh, mtg = 2 * QG * hf + mt;
        float acc[4] = {coff[0], coff[1], coff[2], coff[3]};
        if (VB == 2) {
          const uint32_t w = vw[(tg * (D / 16) + mtg) * 32 + lane];
          const uint32_t w2 = w >> 2, w6 = w >> 6;
          mma_f16(acc, w & 0x00030003u, w2 & 0x00030003u, w & 0x00300030u, w6 & 0x00300030u, bf[0][0], bf[0][1]);
          mma_f16(acc, w & 0x00C000C0u, w6 & 0x00C000C0u, w & 0x03000300u, w6 & 0x03000300u, bf[1][0], bf[1][1]);
        } else {
          const uint2 ww = reinterpret_cast<const uint2*>(vw)[(tg * (D / 16) + mtg) * 32 + lane];
          const uint32_t x0 = ww.x, x8 = ww.x >> 8, y0 = ww.y, y8 = ww.y >> 8;
          mma_f16(acc, x0 & 0x000F000Fu, x8 & 0x000F000Fu, x0 & 0x00F000F0u, x8 & 0x00F000F0u, bf[0][0], bf[0][1]);
          mma_f16(acc, y0 & 0x000F000Fu, y8 & 0x000F000Fu, y0 & 0x00F000F0u, y8 & 0x00F000F0u, bf[1][0], bf[1][1]);
        }
        O[mt][0] = fmaf(O[mt][0], alpha[0], acc[0]);
        O[mt][1] = fmaf(O[mt][1], alpha[1], acc[1]);
        O[mt][2] = fmaf(O[mt][2], alpha[0], acc[2]);
        O[mt][3] = fmaf(O[mt][3], alpha[1], acc[3]);
      }
    }
    // every warp of the stream is done with stage s_ (and with xbuf)
    if (NS == 1) __syncthreads();
    else named_barrier(5 + stream, 32 * SW);
    if (issuer && kt < 0 && ip + NS * STAGES < npg) {
      if (PAGED) {  // branch-free: a page without a block reads block 0 and is reported after the loop
        const int blk = next_blk;  // loaded one page earlier, off this warp's critical path
        if (ip + NS + NS * STAGES < npg) next_blk = lv.btab[(size_t)slot * lv.max_pages + pg0 + ip + NS + NS * STAGES];
        const bool okb = (unsigned)blk < (unsigned)lv.n_blocks;
        bad_block |= !okb;
        mbar_expect_tx(&full[stream * STAGES + s_], PB);
        bulk_g2s(stage0 + (size_t)(stream * STAGES + s_) * PB, lv.pages + ((size_t)(okb ? blk : 0) * lv.Hkv + h) * PB,
                 PB, &full[stream * STAGES + s_]);
      } else {
        mbar_expect_tx(&full[stream * STAGES + s_], PB);
        bulk_g2s(stage0 + (size_t)(stream * STAGES + s_) * PB, gpages + (size_t)(pg0 + ip + NS * STAGES) * PB, PB,
                 &full[stream * STAGES + s_]);
      }
    }
  }
  if (PAGED && bad_block) set_status(lv.status, TQ_DEV_ERR_BLOCK);
  if (__syncthreads_or(kt >= 0)) {
    // A wait gave up. Each stream's issuing thread waits (bounded) for the copies it issued that it has
    // not seen land: its refills stopped at its first failed wait kt, so they are pages kt .. kt + STAGES - 1
    // of the stream (the hook's page was never issued). Only then may the stages be reused below, or the
    // CTA exit. If such a copy still does not land, the CTA leaves its shared memory alone.
    bool drained = true;
    if (issuer && kt >= 0) {
      const int nk = (npg - stream + NS - 1) / NS;
      for (int j = kt; j < kt + STAGES && j < nk; ++j)
        if (!(stream == 0 && j == fault_k)) drained = mbar_wait(&full[stream * STAGES + j % STAGES], (j / STAGES) & 1) && drained;
    }
    if (tid == 0) set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
    if (!__syncthreads_and(drained)) {
      write_empty_partial(part, D, tid, NT, NCOL);
      finish_unit<D, NT, QP>(a, b, h, smem, false);
      return;
    }
  }
  // ---- merge the token groups' partials through shared memory ----
  __syncthreads();
  constexpr int NGRP = 4 * NS;                     // (stream, token group) partials
  const int grp = 4 * stream + tg;
  float* wm = reinterpret_cast<float*>(stage0);  // [NGRP][NCOL query columns]
  float* wl = wm + NCOL * NGRP;                  // [NGRP][NCOL]
  float* wo = wl + NCOL * NGRP;                  // [NGRP][NCOL][D]
  {
    float l0 = l_acc[0], l1 = l_acc[1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    if (hf == 0 && g == 0 && 2 * c < NCOL) {
      wm[grp * NCOL + 2 * c] = m_eff[0];
      wm[grp * NCOL + 2 * c + 1] = m_eff[1];
      wl[grp * NCOL + 2 * c] = l0;
      wl[grp * NCOL + 2 * c + 1] = l1;
    }
    if (2 * c < NCOL) {
#pragma unroll
      for (int mt = 0; mt < 2 * QG; ++mt) {
        const int j0 = CW * hf + 16 * mt + g;
        wo[(grp * NCOL + 2 * c) * D + j0] = O[mt][0];
        wo[(grp * NCOL + 2 * c + 1) * D + j0] = O[mt][1];
        wo[(grp * NCOL + 2 * c) * D + j0 + 8] = O[mt][2];
        wo[(grp * NCOL + 2 * c + 1) * D + j0 + 8] = O[mt][3];
      }
    }
  }
  __syncthreads();
  float* wf = wo + NGRP * NCOL * D;  // [NGRP][NCOL] group weights exp2(m_group - m)
  if (tid < NCOL * NGRP) {
    const int hd = tid % NCOL, w = tid / NCOL;
    float m = -INFINITY;
#pragma unroll
    for (int v = 0; v < NGRP; ++v) m = fmaxf(m, wm[v * NCOL + hd]);
    const float mw = wm[w * NCOL + hd];
    wf[w * NCOL + hd] = (m == -INFINITY || mw == -INFINITY) ? 0.f : exp2f(mw - m);
  }
  __syncthreads();
  for (int i = tid; i < NCOL * D; i += NT) {
    const int hd = i / D, j = i % D;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < NGRP; ++w) o = fmaf(wf[w * NCOL + hd], wo[(w * NCOL + hd) * D + j], o);
    part[2 * NCOL + hd * D + j] = o;
    if (j == 0) {
      float m = -INFINITY, l = 0.f;
#pragma unroll
      for (int w = 0; w < NGRP; ++w) {
        m = fmaxf(m, wm[w * NCOL + hd]);
        l = fmaf(wf[w * NCOL + hd], wl[w * NCOL + hd], l);
      }
      part[hd] = m;
      part[NCOL + hd] = l;
    }
  }
  finish_unit<D, NT, QP>(a, b, h, smem);
}

template <int D, int VB>
constexpr int decode_stages() {  // pages in flight per stream
  return D <= 128 ? 4 : 3;
}

template <int D, int VB, int KB, int QP = 1, int STAGES = decode_stages<D, VB>()>
size_t decode_smem_bytes() {
  const PageLayout pl = page_layout(D, VB, KB);
  constexpr int NT = decode_threads<D>();
  constexpr int NGRP = 4 * decode_streams<D>();
  constexpr int NCOL = qcols<QP>();
  const size_t merge_bytes = sizeof(float) * (3 * NGRP * NCOL + NGRP * NCOL * D);
  const size_t xbuf_bytes = sizeof(float) * decode_xbuf_floats<D>();
  size_t smem = 128 + (size_t)decode_streams<D>() * STAGES * pl.bytes + xbuf_bytes +
                prep_scratch_bytes<D, KB, QP>();
  smem = std::max(smem, 128 + merge_bytes);
  smem = std::max(smem, ring_smem_bytes<D, QP>());
  smem = std::max(smem, 128 + sizeof(float) * (4 * (NT / 32) + 2 * NCOL * 1026));  // combine: split (m, l)
  return smem;
}

// Sets the kernels' shared-memory attributes once and returns resident split-K CTAs per SM.
template <int D, int VB, int KB>
int decode_setup() {
  static int resident = 0;  // set once, outside any stream capture that follows
  if (resident == 0) {
    constexpr int STAGES = decode_stages<D, VB>();
    const size_t smem = decode_smem_bytes<D, VB, KB>();
    if (cudaFuncSetAttribute(k_decode<D, VB, STAGES, false, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(k_decode<D, VB, STAGES, true, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return -1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_decode<D, VB, STAGES, false, KB>, decode_threads<D>(),
                                                      smem) != cudaSuccess ||
        n < 1)
      n = 1;
    resident = n;
  }
  return resident;
}

// Pages in flight per stream of the query-pair (prefill) kernel: the decode's count, or one fewer
// where the pair kernel's shared memory would not fit (head_dim 128 with key_bits 4).
template <int D, int VB, int KB>
constexpr int pair_stages() {
  constexpr int S = decode_stages<D, VB>();
  constexpr size_t page_bytes = (size_t)KB * kPage * D / 8 + 4 * kPage + (size_t)kPage * D * VB / 8 + 2 * kPage * (D / 32);
  return 128 + (size_t)decode_streams<D>() * S * page_bytes + sizeof(float) * decode_xbuf_floats<D>() +
                     prep_scratch_bytes<D, KB, 2>() <= kMaxSmemPerCta
             ? S
             : S - 1;
}

// qp = 2: prefill query pairs (contiguous cache); `batch` is then the number of CTA rows (pairs).
template <int D, int VB, int KB>
cudaError_t launch_decode_dv(const DecodeArgs& a, int batch, int phase, cudaStream_t s, int qp) {
  constexpr int STAGES = decode_stages<D, VB>();
  if (decode_setup<D, VB, KB>() < 0) return cudaErrorInvalidValue;
  constexpr int PSTAGES = pair_stages<D, VB, KB>();
  const size_t smem = qp == 2 ? decode_smem_bytes<D, VB, KB, 2, PSTAGES>() : decode_smem_bytes<D, VB, KB>();
  if (qp == 2) {  // query pairs (prefill): attribute set once, outside any stream capture that follows
    static bool pair_attr = false;
    if (!pair_attr) {
      if (smem > kMaxSmemPerCta) return cudaErrorInvalidValue;
      cudaError_t e = cudaFuncSetAttribute(k_decode<D, VB, PSTAGES, false, KB, 2>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      pair_attr = true;
    }
  }
  if (phase == 0) {  // zero the arrival counters (every decode call leaves them at zero)
    cudaError_t e = cudaMemsetAsync(a.ws + a.plan.cnt_off, 0, sizeof(int32_t) * (size_t)batch * a.lv.Hkv, s);
    if (e != cudaSuccess) return e;
  }
  if (phase < 0 || phase == 1) {
    const dim3 grid(a.plan.n_splits + 1, a.lv.Hkv, batch);
    cudaError_t e =
        qp == 2 ? launch_pdl(k_decode<D, VB, PSTAGES, false, KB, 2>, grid, dim3(decode_threads<D>()), smem, s, a)
        : a.lv.btab ? launch_pdl(k_decode<D, VB, STAGES, true, KB>, grid, dim3(decode_threads<D>()), smem, s, a)
                    : launch_pdl(k_decode<D, VB, STAGES, false, KB>, grid, dim3(decode_threads<D>()), smem, s, a);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;  // phase 2 (combine) runs inside phase 1's last CTA of every (row, KV head)
}

}  // namespace

// True when the query-pair (prefill) kernel of ctx's shape fits the per-CTA shared memory.
bool decode_pairs_fit(const tq_ctx* ctx) {
  const int d = ctx->cfg.head_dim, vb = ctx->cfg.value_bits, kb = ctx->cfg.key_bits;
  size_t b;
  if (kb == 4)
    b = d == 64    ? decode_smem_bytes<64, 4, 4, 2, pair_stages<64, 4, 4>()>()
        : d == 128 ? decode_smem_bytes<128, 4, 4, 2, pair_stages<128, 4, 4>()>()
                   : decode_smem_bytes<256, 4, 4, 2, pair_stages<256, 4, 4>()>();
  else if (d == 64)
    b = vb == 2 ? decode_smem_bytes<64, 2, 3, 2, pair_stages<64, 2, 3>()>()
                : decode_smem_bytes<64, 4, 3, 2, pair_stages<64, 4, 3>()>();
  else if (d == 128)
    b = vb == 2 ? decode_smem_bytes<128, 2, 3, 2, pair_stages<128, 2, 3>()>()
                : decode_smem_bytes<128, 4, 3, 2, pair_stages<128, 4, 3>()>();
  else
    b = vb == 2 ? decode_smem_bytes<256, 2, 3, 2, pair_stages<256, 2, 3>()>()
                : decode_smem_bytes<256, 4, 3, 2, pair_stages<256, 4, 3>()>();
  return b <= kMaxSmemPerCta;
}

// key_bits 4 is served with value_bits 4 (validated on the host).
int decode_resident_ctas(const tq_ctx* ctx) {
  const int d = ctx->cfg.head_dim, vb = ctx->cfg.value_bits, kb = ctx->cfg.key_bits;
  int n;
  if (kb == 4) n = d == 64 ? decode_setup<64, 4, 4>() : d == 128 ? decode_setup<128, 4, 4>() : decode_setup<256, 4, 4>();
  else if (d == 64 && vb == 2) n = decode_setup<64, 2, 3>();
  else if (d == 64 && vb == 4) n = decode_setup<64, 4, 3>();
  else if (d == 128 && vb == 2) n = decode_setup<128, 2, 3>();
  else if (d == 128 && vb == 4) n = decode_setup<128, 4, 3>();
  else if (d == 256 && vb == 2) n = decode_setup<256, 2, 3>();
  else n = decode_setup<256, 4, 3>();
  return n > 0 ? n : 1;
}

cudaError_t launch_decode(const tq_ctx* ctx, int layer, const void* q, float* out, const int32_t* seq_ids,
                          int batch, float scale, void* ws, const DecodePlan& plan, int phase, cudaStream_t s, int qpr,
                          const int32_t* n_q, int qp) {
  if (qp == 2 && (qpr % 2 != 0 || ctx->cfg.n_blocks > 0)) return cudaErrorInvalidValue;
  DecodeArgs a;
  a.lv = layer_view(ctx, layer);
  a.qpr = qpr;
  a.n_q = n_q;
  a.q = static_cast<const uint16_t*>(q);
  a.out = out;
  a.seq_ids = seq_ids;
  a.scale = scale;
  a.ws = static_cast<uint8_t*>(ws);
  a.plan = plan;
  a.fault_stage = g_fault_stage.load();
  a.fault_polls = (uint32_t)g_fault_polls.load();
  const int d = ctx->cfg.head_dim, vb = ctx->cfg.value_bits, kb = ctx->cfg.key_bits;
  if (kb == 4) {
    if (d == 64) return launch_decode_dv<64, 4, 4>(a, batch, phase, s, qp);
    if (d == 128) return launch_decode_dv<128, 4, 4>(a, batch, phase, s, qp);
    return launch_decode_dv<256, 4, 4>(a, batch, phase, s, qp);
  }
  if (d == 64 && vb == 2) return launch_decode_dv<64, 2, 3>(a, batch, phase, s, qp);
  if (d == 64 && vb == 4) return launch_decode_dv<64, 4, 3>(a, batch, phase, s, qp);
  if (d == 128 && vb == 2) return launch_decode_dv<128, 2, 3>(a, batch, phase, s, qp);
  if (d == 128 && vb == 4) return launch_decode_dv<128, 4, 3>(a, batch, phase, s, qp);
  if (d == 256 && vb == 2) return launch_decode_dv<256, 2, 3>(a, batch, phase, s, qp);
  return launch_decode_dv<256, 4, 3>(a, batch, phase, s, qp);
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
// For them this variant takes only inputs and outputs. Its scratch (split partials and arrival
// counters) lives in the file-scope device array below, so it has a fixed maximum size.
// =============================================================================================
namespace tq {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB, held by every device that loads libtq
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
// The arrival counters sit in a fixed region at the start of the array, one per (row, KV head), and the
// split partials start right after it, whatever the context. Calls on contexts of different shapes
// therefore never place one context's partials over another's counters (the workspace plan of a
// context sizes its counter region by that context's max_seqs x n_kv_heads).
constexpr size_t kNoAllocCounters = 16384;

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
  if ((size_t)batch * ctx->cfg.n_kv_heads > tq::kNoAllocCounters)
    return tq::set_error(TQ_ERR_CAPACITY, "batch x n_kv_heads exceeds the 16384 arrival counters of the built-in "
                                          "scratch of tq_decode_attention_noalloc");
  tq::DecodePlan plan = tq::decode_plan(ctx, batch, max_ctx_hint);
  plan.cnt_off = 0;
  plan.part_off = tq::kNoAllocCounters * sizeof(int32_t);
  plan.bytes = (plan.part_off + plan.part_stride * (size_t)batch * ctx->cfg.n_kv_heads * (plan.n_splits + 1) + 255) /
               256 * 256;
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

extern "C" tq_status tq_debug_decode_wait_fault(int stage, int polls) {
  if (stage < -1 || stage > 3) return tq::set_error(TQ_ERR_INVALID_ARG, "stage must be -1 (off) or 0..3");
  if (stage >= 0 && (polls < 1 || polls > (int)tq::kWaitPolls))
    return tq::set_error(TQ_ERR_INVALID_ARG, "polls must be in [1, 2^22]");
  tq::g_fault_polls.store(stage >= 0 ? polls : 0);
  tq::g_fault_stage.store(stage);
  return tq::set_error(TQ_OK, "");
}
