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

#include "tq_decode_common.cuh"
#include "tq_quantize_common.cuh"

namespace tq {
namespace {

// Wait-timeout test hook (tq_debug_decode_wait_fault), read by every decode launch.
std::atomic<int> g_fault_stage{-1};
std::atomic<int> g_fault_polls{0};

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
// Decode step: the new token has filled the ring of (row b, KV head h) to 128 tokens (L, the length
// with it, is a multiple of 128). The ring CTA codes those 128 tokens into their packed page now, so
// that the step whose token starts the next ring block finds every block below it coded (appends keep
// the same rule). The tokens are the ring rows before the new one and the new token from the input.
template <int D, int KB, int NT>
__device__ __noinline__ void step_code_block(const DecodeArgs& a, int b, int h, int slot, int L, uint8_t* smem) {
  AppendArgs ap;
  ap.lv = a.lv;
  ap.k = a.k_new;
  ap.v = a.v_new;
  ap.dt = a.new_dt;
  ap.seq_ids = a.seq_ids;
  ap.n_new = nullptr;
  ap.max_new = 1;
  ap.flush = 0;
  ap.full = 0;
  const int Np = L - kPage;  // the ring's first position
  for (int q32 = 0; q32 < 4; ++q32) {
    __syncthreads();  // shared memory is free: the ring split and combine, or the previous block, are done
    quantize_page_cta<D, KB, NT>(ap, b, h, slot, L - 1, Np, Np / kPage, kPage, q32, smem);
  }
}

template <int D, int VB, int STAGES, bool PAGED, int KB, int QP = 1, bool WIDE = false>
__global__ void __launch_bounds__(decode_threads<D, WIDE>(), (D == 256 && VB == 2) || WIDE ? 2 : 1)
    k_decode(DecodeArgs a) {
  constexpr int NCOL = qcols<QP>();
  constexpr int NBP = key_loop_planes(KB, D, QP);  // B planes the key MMAs run (stored planes: KB)
  constexpr int RP = key_rem_plane(KB, D);
  constexpr bool REMN = key_rem_in_n(KB, D, QP);   // the remainder sits in columns 4..7 of plane 0
  constexpr int CW = warp_coords<D>();  // coordinates per warp
  constexpr int HALVES = D / CW;
  constexpr int KS = CW / 16;           // key-MMA k-steps per warp
  constexpr int QG = CW / 32;           // value groups per warp
  constexpr int NT = decode_threads<D, WIDE>();
  constexpr int NS = decode_streams<D, WIDE>();
  constexpr int SW = 4 * HALVES;  // warps per stream
  constexpr int NG = D / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const LayerView& lv = a.lv;
  const int sp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int stream = warp / SW, tg = warp & 3, hf = (warp % SW) >> 2;
  const int nsp = a.plan.n_splits;
  if (a.late_state) pdl_wait();  // the previous launch was a decode step of this layer: see DecodeArgs
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
    finish_unit<D, NT, QP>(a, b, h, reinterpret_cast<float*>(smem + 128));
    return;
  }
  if (sp == nsp) {
    pdl_wait();
    pdl_launch();
    int L1 = 0, Np1, P1;
    bool stepped = false;
    if (QP == 1 && a.k_new) seq_view(a, slot, L1, Np1, P1, stepped);  // before this unit can finish
    const bool smem_ok = ring_split<D, NT, QP>(a, b, h, slot, part, smem);
    finish_unit<D, NT, QP>(a, b, h, reinterpret_cast<float*>(smem + 128), smem_ok);
    if (QP == 1 && stepped && smem_ok && L1 % kPage == 0) step_code_block<D, KB, NT>(a, b, h, slot, L1, smem + 128);
    return;
  }
  int L, Np, P;
  bool stepped;
  seq_view(a, slot, L, Np, P, stepped);
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
    finish_unit<D, NT, QP>(a, b, h, reinterpret_cast<float*>(smem + 128));
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
        // column h + 4 (lanes c ^ 2) holds the remainder part of head h
        if (REMN) am[i] += __shfl_xor_sync(0xffffffffu, am[i], 2);
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
      finish_unit<D, NT, QP>(a, b, h, reinterpret_cast<float*>(smem + 128), false);
      return;
    }
  }
  // ---- merge the token groups' partials through shared memory ----
  __syncthreads();
  constexpr int NGRP = 4 * NS;                     // (stream, token group) partials
  const int grp = 4 * stream + tg;
  float* wm = reinterpret_cast<float*>(stage0);  // [NGRP][NCOL query columns]
  float* wl = wm + NCOL * NGRP;                  // [NGRP][NCOL]
  float* wo = wl + NCOL * NGRP;                  // [NGRP][NCOL][D + 4] (rows padded: the c lanes meet other banks)
  constexpr int WS = D + 4;
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
        wo[(grp * NCOL + 2 * c) * WS + j0] = O[mt][0];
        wo[(grp * NCOL + 2 * c + 1) * WS + j0] = O[mt][1];
        wo[(grp * NCOL + 2 * c) * WS + j0 + 8] = O[mt][2];
        wo[(grp * NCOL + 2 * c + 1) * WS + j0 + 8] = O[mt][3];
      }
    }
  }
  __syncthreads();
  // each output element takes the groups' maximum and weights exp2(m_group - m) itself (no third barrier)
  for (int i = tid; i < NCOL * D; i += NT) {
    const int hd = i / D, j = i % D;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < NGRP; ++w) m = fmaxf(m, wm[w * NCOL + hd]);
    float o = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < NGRP; ++w) {
      const float mw = wm[w * NCOL + hd];
      const float f = (m == -INFINITY || mw == -INFINITY) ? 0.f : exp2f(mw - m);
      o = fmaf(f, wo[(w * NCOL + hd) * WS + j], o);
      l = fmaf(f, wl[w * NCOL + hd], l);
    }
    part[2 * NCOL + hd * D + j] = o;
    if (j == 0) {
      part[hd] = m;
      part[NCOL + hd] = l;
    }
  }
  finish_unit<D, NT, QP>(a, b, h, reinterpret_cast<float*>(smem + 128));
}

template <int D, int VB>
constexpr int decode_stages() {  // pages in flight per stream
  return D <= 128 ? 4 : 3;
}

template <int D, int VB, int KB, int QP = 1, int STAGES = decode_stages<D, VB>(), bool WIDE = false>
size_t decode_smem_bytes() {
  const PageLayout pl = page_layout(D, VB, KB);
  constexpr int NT = decode_threads<D, WIDE>();
  constexpr int NGRP = 4 * decode_streams<D, WIDE>();
  constexpr int NCOL = qcols<QP>();
  const size_t merge_bytes = sizeof(float) * (3 * NGRP * NCOL + NGRP * NCOL * (D + 4));
  const size_t xbuf_bytes = sizeof(float) * decode_xbuf_floats<D>();
  size_t smem = 128 + (size_t)decode_streams<D, WIDE>() * STAGES * pl.bytes + xbuf_bytes +
                prep_scratch_bytes<D, KB, QP, NT>();
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

// The WIDE variant (head_dim 128, K3/V2, contiguous cache): attributes set once; resident CTAs per SM.
int decode_setup_wide() {
  static int resident = 0;  // set once, outside any stream capture that follows
  if (resident == 0) {
    constexpr int STAGES = decode_stages<128, 2>();
    const size_t smem = decode_smem_bytes<128, 2, 3, 1, STAGES, true>();
    if (cudaFuncSetAttribute(k_decode<128, 2, STAGES, false, 3, 1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return -1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_decode<128, 2, STAGES, false, 3, 1, true>,
                                                      decode_threads<128, true>(), smem) != cudaSuccess ||
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
    if constexpr (D == 128 && VB == 2 && KB == 3) {
      if (a.plan.wide && qp == 1 && !a.lv.btab) {  // decode_plan chose the two-CTAs-per-SM variant
        if (decode_setup_wide() < 0) return cudaErrorInvalidValue;
        return launch_pdl(k_decode<128, 2, STAGES, false, 3, 1, true>, grid, dim3(decode_threads<128, true>()),
                          decode_smem_bytes<128, 2, 3, 1, STAGES, true>(), s, a);
      }
    }
    cudaError_t e =
        qp == 2 ? launch_pdl(k_decode<D, VB, PSTAGES, false, KB, 2>, grid, dim3(decode_threads<D>()), smem, s, a)
        : a.lv.btab ? launch_pdl(k_decode<D, VB, STAGES, true, KB>, grid, dim3(decode_threads<D>()), smem, s, a)
                    : launch_pdl(k_decode<D, VB, STAGES, false, KB>, grid, dim3(decode_threads<D>()), smem, s, a);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;  // the combine runs inside phase 1's last CTA of every (row, KV head)
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
int decode_resident_ctas(const tq_ctx* ctx, bool wide) {
  const int d = ctx->cfg.head_dim, vb = ctx->cfg.value_bits, kb = ctx->cfg.key_bits;
  int n;
  if (wide) {
    n = decode_setup_wide();
    return n > 0 ? n : 1;
  }
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
                          const int32_t* n_q, int qp, const void* k_new, const void* v_new, int new_dt, int late_state) {
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
  a.k_new = k_new;
  a.v_new = v_new;
  a.new_dt = new_dt;
  a.late_state = late_state;
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
  const tq::NvtxRange nvtx_range("tq_decode_attention_noalloc");
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
  plan.row_cnt_off = 0;  // no decode step runs on this scratch
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
  e = tq::launch_decode(ctx, layer, q, out, d_seq_ids, batch, scale, scratch, plan, -1, (cudaStream_t)stream, 1,
                        nullptr, 1, nullptr, nullptr, 0, tq::step_follows(ctx, layer, (cudaStream_t)stream) ? 1 : 0);
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
