// Device code of the decode kernels that is not their page loop: arguments, MMA helpers, query rotation and
// projection, the exact ring split, the cross-split combine and the arrival protocol.
#pragma once

#include <cmath>

#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {

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
  // Decode step (tq_decode_step): one new token per row, k_new / v_new [B][Hkv][D] (bf16, or fp32 when
  // new_dt = 1), is appended by this launch and attended to. nullptr for a plain decode.
  const void* k_new;
  const void* v_new;
  int new_dt;
  // 1: the previous launch on the stream was a decode step of this layer, which changes the sequence
  // state and may code a page after it released its dependents; this launch then reads the state and
  // pages only after its stream wait.
  int late_state;
};

namespace {

constexpr float kLog2e = 1.4426950408889634f;
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


// The sequence as a decode CTA sees it: L tokens, of which the first Np lie in packed blocks before
// the ring and P = Np + F are read packed (F: ring tokens a flush coded). In a decode step the row is
// seen with its new token (stepped; a row already at max_ctx takes none and is decoded as it stands).
// Every CTA of a row reads the state before any of them can change it (the row's length is published
// by the last (row, KV head) unit to finish, see row_arrive).
__device__ __forceinline__ void seq_view(const DecodeArgs& a, int slot, int& L, int& Np, int& P, bool& stepped) {
  const LayerView& lv = a.lv;
  L = lv.state[2 * slot];
  int F = lv.state[2 * slot + 1];
  const int Np0 = L > 0 ? kPage * ((L - 1) / kPage) : 0;
  stepped = a.k_new != nullptr && L < lv.max_ctx;
  if (stepped) ++L;
  Np = L > 0 ? kPage * ((L - 1) / kPage) : 0;
  if (Np != Np0) F = 0;  // the new token starts a new ring block
  P = Np + F;
}

// One element of the step's new token (K: which = 0, V: 1) as bf16 bits, as an append stores it.
__device__ __forceinline__ uint16_t new_token_elem(const DecodeArgs& a, int which, int b, int h, int j) {
  const size_t i = ((size_t)b * a.lv.Hkv + h) * a.lv.d + j;
  const void* base = which ? a.v_new : a.k_new;
  return a.new_dt ? f32_to_bf16_rn(static_cast<const float*>(base)[i]) : static_cast<const uint16_t*>(base)[i];
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

template <int D, bool WIDE = false>
__host__ __device__ constexpr int decode_threads();
// Floats of the d=256 partial-score exchange buffer of a split CTA ([NT][2 tiles][8]).
template <int D>
__host__ __device__ constexpr int decode_xbuf_floats() {
  return D == 256 ? decode_threads<D>() * 2 * 8 : 0;
}

// Split CTAs run `decode_streams` independent page streams of 4 token-group warps x (d/128) coordinate
// halves: 3 streams (12 warps, one CTA per SM) for head_dim 128, 1 stream (8 warps) for head_dim 256.
// (Four streams of 16 warps measured slower at batch 1 and no faster at batch 32.) The WIDE variant of
// head_dim 128 (K3/V2, contiguous cache) runs 2 streams in CTAs of which two share an SM: at batch 32 x
// 128K it hides more latency (1145 against 1205 us per launch); at batch 1 its extra splits cost more.
template <int D, bool WIDE = false>
__host__ __device__ constexpr int decode_streams() {
  return D <= 128 ? (WIDE ? 2 : 3) : 1;
}
// Coordinates of one warp (a 128-coordinate half, or all 64) and key-MMA k-steps per warp.
template <int D>
__host__ __device__ constexpr int warp_coords() {
  return D < 128 ? D : 128;
}
template <int D, bool WIDE>
__host__ __device__ constexpr int decode_threads() {
  return decode_streams<D, WIDE>() * 32 * 4 * (D / warp_coords<D>());
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
// With one query row per CTA (decode), B columns 4..7 of the MMAs are free: the remainder plane then rides in
// plane 0's MMAs as columns 4..7 (column 4 + h = the remainder of head h), and the epilogue adds column
// 4 + h to column h. No MMA, mask or load is spent on it. B planes that the page loop runs:
__host__ __device__ constexpr bool key_rem_in_n(int kb, int d, int qp) { return qp == 1 && key_rem_plane(kb, d) >= 0; }
__host__ __device__ constexpr int key_loop_planes(int kb, int d, int qp) {
  return key_bplanes(kb, d) - (key_rem_in_n(kb, d, qp) ? 1 : 0);
}

// Query columns of a split CTA: the 8 B columns of the MMAs carry the kMaxG heads of QP query rows
// (QP = 1 for decode; 2 for prefill, whose chunk queries of one sequence share the key operands).
template <int QP>
__host__ __device__ constexpr int qcols() {
  return kMaxG * QP;
}

// Bytes of a split CTA's query-prep scratch.
template <int D, int KB, int QP = 1, int NT = decode_threads<D>()>
__host__ __device__ constexpr size_t prep_scratch_bytes() {
  // q_rot, q_proj [columns][D] fp32; 32 floats of scales; B fragments [planes D/16 items][32 lanes]
  // uint2; per-warp offset sums [warps][2][8 B columns]
  return sizeof(float) * (2 * qcols<QP>() * D + 32) + 8 * 32 * (key_loop_planes(KB, D, QP) * D / 16) +
         sizeof(float) * 2 * 8 * (NT / 32);
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
// q_rot = Pi q (a warp per query column: FWHT with the signs D) and q_proj = S q_rot (m16n8k16 with A = S
// in f16 from the tables and B = q_rot split into f16 hi + lo), for the NCOL query columns of (row b, KV
// head h); zero columns for heads >= G. Writes qr, qp [NCOL][D] and, per column, red[col] (the power of two
// that scaled q_rot for the f16 projection) and red[3 NCOL + col] = max |q_rot|. All NT threads; ends with
// a block barrier.
template <int D, int NT, int QP>
__device__ __forceinline__ void query_rot_proj(const DecodeArgs& a, int b, int h, float* qr, float* qp, float* red,
                                               const SFrag<D>& sf) {
  constexpr int NCOL = qcols<QP>();
  constexpr int NE = D / 32;
  constexpr int MT = D / 16;
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int G = lv.G;
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
      red[warp] = mx > 0.f ? exp2f(floorf(log2f(16384.f / mx))) : 1.f;
      red[3 * NCOL + warp] = mx;
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
}

template <int D, int NT, int KB, int QP = 1>
__device__ __forceinline__ void query_prep(const DecodeArgs& a, int b, int h, float* ps, const SFrag<D>& sf,
                                           float (&um)[2], float (&cm)[2], float (&uq)[2], float (&cq)[2]) {
  constexpr int NCOL = qcols<QP>();
  constexpr int NBP = key_bplanes(KB, D), QJP = key_qjl_plane(KB), RP = key_rem_plane(KB, D);
  constexpr int NMW = KB == 3 ? 2 : 4;  // index-plane weights
  constexpr int HALVES = D / warp_coords<D>();
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int G = lv.G;
  float* qr = ps;              // [NCOL][D]
  float* qp = qr + NCOL * D;   // [NCOL][D]
  float* red = qp + NCOL * D;  // [col]: projection lambda; [NCOL + 2 col + {0, 1}]: operand lambdas; [3 NCOL + col]: max
  query_rot_proj<D, NT, QP>(a, b, h, qr, qp, red, sf);
  if (tid < NCOL) {  // operand lambdas of column tid
    float wmax = 0.f;  // largest |2 w| of the index planes
#pragma unroll
    for (int p = 0; p < NMW; ++p) wmax = fmaxf(wmax, fabsf(2.f * lv.cb[kCbW + p]));
    const float mx = red[3 * NCOL + tid];
    const float big = 16777216.f;  // 2^24, the largest bit-plane prescale
    const float bm = wmax * mx * big, bp = 2.f * lv.cb[kCbSmax] * mx * big;
    red[NCOL + 2 * tid + 0] = bm > 0.f ? exp2f(floorf(log2f(32768.f / bm))) : 1.f;
    red[NCOL + 2 * tid + 1] = bp > 0.f ? exp2f(floorf(log2f(32768.f / bp))) : 1.f;
  }
  __syncthreads();
  // B fragments: item (hv, pi, s) is computed by warp item % NW and shared through shared memory;
  // wsum[w][n] / wsum[w][8 + n] hold warp w's offset sums of B column n, added in a fixed order below
  // (the same constants in every split CTA and every call)
  constexpr int KS = warp_coords<D>() / 16;  // key-MMA k-steps per warp
  constexpr bool REMN = key_rem_in_n(KB, D, QP);  // the remainder rides in columns 4..7 of plane 0
  constexpr int NBPL = key_loop_planes(KB, D, QP);
  constexpr int NW = NT / 32, NITEMS = HALVES * NBPL * KS;
  uint2* frag = reinterpret_cast<uint2*>(red + 32);  // [NITEMS][32]
  float* wsum = reinterpret_cast<float*>(frag + NITEMS * 32);  // [NW][2][8]
  const bool rem_lane = REMN && g >= kMaxG;  // B column g carries the remainder of head g - 4
  const int hsrc = rem_lane ? g - kMaxG : g;
  const bool live = hsrc < NCOL && hsrc % kMaxG < G;
  const float lam_m = live ? red[NCOL + 2 * hsrc] : 0.f, lam_q = live ? red[NCOL + 2 * hsrc + 1] : 0.f;
  const float* bm = qr + (live ? hsrc : 0) * D;
  const float* bp = qp + (live ? hsrc : 0) * D;
  __syncthreads();
  float sum_m = 0.f, sum_q = 0.f;
  for (int item = warp; item < NITEMS; item += NW) {
    const int s = item % KS, pi = (item / KS) % NBPL, hv = item / (NBPL * KS);
    const bool qjl = pi == QJP;
    // rem: this lane's operand is the remainder of plane 0 (a remainder plane, or columns 4..7 of plane 0)
    const bool rem = REMN ? (rem_lane && pi == 0) : pi == RP;
    const float w = (rem_lane && pi != 0) ? 0.f
                    : qjl                 ? 2.f * lam_q
                                          : 2.f * lv.cb[kCbW + (rem ? 0 : pi)] * lam_m;
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
  if (c == 0) {
    wsum[warp * 16 + g] = sum_m;
    wsum[warp * 16 + 8 + g] = sum_q;
  }
  __syncthreads();
  const float kappa = 1.2533141373155003f / (float)D;  // sqrt(pi/2) / d
#pragma unroll
  for (int i = 0; i < 2; ++i) {  // C-fragment column 2c + i is query column hd
    const int hd = min(2 * c + i, NCOL - 1);
    float sm = 0.f, sq = 0.f;
    for (int w = 0; w < NW; ++w) {
      sm += wsum[w * 16 + hd] + (REMN ? wsum[w * 16 + kMaxG + hd] : 0.f);
      sq += wsum[w * 16 + 8 + hd];
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
  bool stepped;
  seq_view(a, slot, L, Np, P, stepped);
  // ring tokens are positions P .. Lq - 1 of each query row
  const int n0 = row_len(a, QP * b, L) - P, n1 = QP == 1 ? n0 : row_len(a, QP * b + 1, L) - P;
  const int F = P - Np, n = max(n0, n1);
  if (n <= 0) {
    write_empty_partial(part, D, tid, NT, NCOL);
    return true;
  }
  // a decode step's new token is ring row n - 1: it comes from the input (and is written to the ring
  // here); the rows before it come from the ring
  const int nm = stepped ? n - 1 : n;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw);
  const uint16_t* krows = reinterpret_cast<const uint16_t*>(smem_raw + 128);  // [n][D] bf16
  const uint16_t* vrows = KV ? krows + (size_t)kPage * D : krows;             // [n][D] bf16
  float* sc = reinterpret_cast<float*>(smem_raw + 128 + (KV ? 2 : 1) * 2 * kPage * D);  // [128][NCOL]
  float* red = sc + kPage * NCOL;                                                        // [NCOL][2] (+ pad)
  float* qs = red + 4 * NCOL;                                                            // [NCOL][D]
  const uint16_t* rk = lv.ring + (((size_t)slot * lv.Hkv + h) * 2) * kPage * D + (size_t)F * D;
  const uint16_t* rv = rk + (size_t)kPage * D;
  const uint32_t bytes = (uint32_t)nm * D * 2;
  if (tid == 0) {
    mbar_init(bar, 1);
    if (KV) mbar_init(bar + 1, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    if (bytes) {
      mbar_expect_tx(bar, bytes);
      bulk_g2s(smem_raw + 128, rk, bytes, bar);
    } else {
      mbar_arrive(bar);
    }
    if (KV) {
      if (bytes) {
        mbar_expect_tx(bar + 1, bytes);
        bulk_g2s(smem_raw + 128 + 2 * kPage * D, rv, bytes, bar + 1);
      } else {
        mbar_arrive(bar + 1);
      }
    }
  }
  if (QP == 1 && stepped) {  // the new token: shared-memory row nm (V later when it shares K's rows) and the ring
    uint16_t* kr = reinterpret_cast<uint16_t*>(smem_raw + 128) + (size_t)nm * D;
    uint16_t* gk = lv.ring + ((((size_t)slot * lv.Hkv + h) * 2) * kPage + F + nm) * D;
    for (int j = tid; j < D; j += NT) {
      const uint16_t kv = new_token_elem(a, 0, b, h, j), vv = new_token_elem(a, 1, b, h, j);
      kr[j] = kv;
      gk[j] = kv;
      gk[(size_t)kPage * D + j] = vv;
      if (KV) kr[(size_t)kPage * D + j] = vv;  // the V rows follow the K rows
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
    if (bytes) {
      mbar_expect_tx(bar, bytes);
      bulk_g2s(smem_raw + 128, rv, bytes, bar);
    } else {
      mbar_arrive(bar);
    }
  }
  if (!KV && QP == 1 && stepped) {  // the new token's V row, where its K row was
    uint16_t* vr = reinterpret_cast<uint16_t*>(smem_raw + 128) + (size_t)nm * D;
    for (int j = tid; j < D; j += NT) vr[j] = new_token_elem(a, 1, b, h, j);
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
// merges all of them (an arrival counter; no CTA waits on another), with `scratch` (shared memory, room
// for 4 (NT/32) + 2 NCOL 1026 floats) as its working space. smem_ok = false: this CTA's shared memory may
// still receive a copy, so a last CTA writes zeros instead of combining.
// Decode step: the last (row, KV head) unit of a row to finish publishes the row's new length (and a
// new ring block's F = 0). Every CTA of the row has read the old state by then: a unit finishes only
// after all of its CTAs arrived, and they read the state before arriving. The per-row counters follow
// the per-unit ones in the workspace and are left at zero.
__device__ __noinline__ void row_arrive(const DecodeArgs& a, int b) {
  int* rc = reinterpret_cast<int*>(a.ws + a.plan.row_cnt_off) + b;
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;\n" : "=r"(old) : "l"(rc) : "memory");
  if (old != a.lv.Hkv - 1) return;
  *rc = 0;
  const LayerView& lv = a.lv;
  const int slot = a.seq_ids[b];
  if (slot < 0 || slot >= lv.max_seqs) {
    set_status(lv.status, TQ_DEV_ERR_SEQ_ID);
    return;
  }
  const int L = lv.state[2 * slot];
  if (L >= lv.max_ctx) {
    set_status(lv.status, TQ_DEV_ERR_CAPACITY);
    return;
  }
  const int Np = L > 0 ? kPage * ((L - 1) / kPage) : 0, Np2 = kPage * (L / kPage);
  lv.state[2 * slot] = L + 1;
  if (Np2 != Np) lv.state[2 * slot + 1] = 0;
}

template <int D, int NT, int QP = 1>
__device__ __noinline__ void finish_unit(const DecodeArgs& a, int b, int h, float* scratch, bool smem_ok = true) {
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
  // The row's arrival does not depend on the merge: the first thread after the merging warps takes it while
  // they merge (the merge has no block barrier).
  constexpr int kArriveTid = 32 * qcols<QP>();
  static_assert(QP != 1 || NT > kArriveTid, "a thread outside the merging warps");
  if (QP == 1 && a.k_new && threadIdx.x == kArriveTid) row_arrive(a, b);
  if (!smem_ok) zero_unit_out<D, NT, QP>(a, b, h);
  else combine_unit<D, NT, QP>(a, b, h, scratch);
}

}  // namespace
}  // namespace tq
