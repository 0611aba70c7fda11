// Prefill attention over the packed history on tcgen05 tensor cores (TurboQuant vLLM guide §七, first
// item: prefill that reads the quantised cache; §三 hybrid estimator, §二 codes). A prefill chunk gives
// every KV head n_q x G query rows against the same packed pages. Here each page is expanded once per
// launch (k_prefill_expand) into the f16 B tiles of the score and P.V MMAs, in the layout the tensor
// cores read, and every tile of 128 query rows (32 queries x the 4 query heads of one KV head) copies
// them into shared memory, instead of by the 8 query columns of the decode kernel's mma.sync path.
//
// One CTA = one tile, one KV head, one split of the tile's visible pages. It writes one partial per
// (query, KV head, split) in the decode workspace's layout (m, l, o in the rotated basis, log2 units);
// k_prefill_ring then adds the exact ring tokens and combines, one small CTA per (query, KV head).
//
// Scores, with the odd-symmetric 2-bit codebook c[idx] = a_h (2 h - 1) + a_l (2 l - 1) and the QJL
// sign s = 2 sigma - 1, are one fp32 accumulator in TMEM:
//   S[r][t] = A_hi . B_h + A_lo . B_h + A_l . B_l + A_qp . B_s
//     A_hi + A_lo = lambda a_h q_rot (f16 hi + remainder), A_l = lambda a_l q_rot, A_qp = lambda kappa
//     (S q_rot) (f16), B_h = B_l = +-1, B_s = +-gamma_t (gamma_t is stored as f16, so exactly),
// so S = lambda (<q_rot, c[idx_t]> + kappa gamma_t <S q_rot, s_t>) up to the f16 rounding of the l and
// QJL operands (as in the decode kernel), and the logit is S n_t scale / lambda. lambda, a power of two
// per tile, keeps the operands inside the f16 range. P (f16) and the dequantised values V^T =
// s_g (code - offset) (f16) feed the P.V MMA into a second TMEM accumulator; the softmax rescales it
// lazily (only when a row maximum grows by more than 2^8).
#include <atomic>
#include <cmath>

#include <cuda_runtime.h>

#include "tq_tcgen05.cuh"

namespace tq {

// tq_debug_prefill_wait_fault: the page (index within its split) whose copy CTA (0, 0, 0) of the tcgen05
// prefill skips (-1: none), and the polls of its wait
std::atomic<int> g_pfault_page{-1};
std::atomic<int> g_pfault_polls{0};

namespace {

// 16 worker warps (warp w covers TMEM lanes 32 (w % 4).. and column quarter w / 4) and one more warp whose
// lane 0 issues every copy and MMA and polls the barriers
constexpr int kPtWorkers = 512, kPtThreads = kPtWorkers + 32, kPtIssuer = kPtWorkers;
constexpr int kPtQ = kPtWorkers / 128;  // column quarters: 32 columns (and 32 coordinates of a row) per thread
// Shared memory (offsets from a 1024-byte aligned base): six 32 KB operand tiles that rotate through the
// page pipeline (the h, l and QJL planes of the scores, V^T, and P over the h plane), then n_t of the pages
// in flight [2][128], the row exchange [4][128], the per-warp operand maxima [16], the barriers and the
// TMEM address.
constexpr uint32_t kPtTileBytes = (uint32_t)kPxTileBytes, kPtSlots = 6, kPtTail0 = kPtSlots * kPtTileBytes;
constexpr uint32_t kPtTail = 2 * 128 * 4 + 4 * 128 * 4 + 16 * 4 + 8 * 8 + 8;
// barriers: S table, projection, the h / l tiles and n_t of a page (two, by page parity), its QJL / V^T
// tiles, score MMAs (QJL part; the h and l part has its own), P.V MMAs
enum { kBarTab = 0, kBarProj = 1, kBarA = 2, kBarB = 4, kBarS = 5, kBarO = 6, kBarHL = 7, kNumBars = 8 };
// TMEM (512 columns): scores S at 0, output O at 128, and from 256 the four f16 A tiles of the scores, 64
// columns each: lambda a_h q_rot (f16 hi), its remainder, lambda a_l q_rot, lambda kappa S q_rot
constexpr uint32_t kPtTmS = 0, kPtTmO = 128, kPtTmA = 256;

struct PrefillTcArgs {
  LayerView lv;
  const uint16_t* q;       // bf16 [batch][qpr][Hq][128]
  const int32_t* seq_ids;  // [batch]
  const int32_t* n_q;      // [batch]: the row's last n_q tokens are its queries
  int qpr;                 // query slots per batch row
  float scale;             // softmax scale
  uint8_t* ws;
  DecodePlan plan;         // partial layout (n_splits history splits per unit), expanded pages
  int fault_page;          // wait-timeout test hook: CTA (0, 0, 0) issues no copy of this page's h / l tiles
  uint32_t fault_polls;    // and gives up its wait for them after this many polls
};

constexpr size_t prefill_tc_smem() { return 1024 + kPtTail0 + kPtTail; }
// the expansion kernel: half an expanded page (two tiles and n_t), then the packed page (at most K3/V4's
// 15872 B) and its barrier
constexpr size_t prefill_expand_smem() { return 1024 + 2 * kPxTileBytes + 512 + 15872 + 16; }
static_assert(2 * (prefill_expand_smem() + 1024) <= 233472, "two expansion CTAs per SM");
static_assert(prefill_tc_smem() <= 232448 && prefill_expand_smem() <= 232448, "shared memory");

// Address of page pg of (slot, KV head h); a paged cache's page without a valid block reads block 0 and
// is reported (TQ_DEV_ERR_BLOCK), as in the decode kernel.
__device__ __forceinline__ const uint8_t* pt_page(const LayerView& lv, int slot, int h, int pg) {
  const uint8_t* p = page_addr(lv, slot, h, pg);
  if (!p) {
    set_status(lv.status, TQ_DEV_ERR_BLOCK);
    p = lv.pages;
  }
  return p;
}

// 2^x (the PTX approximate base-2 exponential; 2^-inf = 0).
__device__ __forceinline__ float pt_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Pairs of f16 (512 + code) from a value word: the code field at bit `pos` (and pos + 16) moved to
// mantissa bits 1.. of an f16 whose exponent puts 0.5 in the last mantissa bit.
template <int VB>
__device__ __forceinline__ uint32_t code_pair_512(uint32_t w, int pos) {
  constexpr uint32_t mask = VB == 2 ? 0x00030003u : 0x000F000Fu;
  return (((w >> pos) & mask) << 1) | 0x60006000u;
}

// One +-c plane of a page into a B tile: token tk's 32 coordinates of quarter hv (4 chunks of 8), from its
// four KBITS words of plane p; a set bit gives +c, a clear one -c (c in both f16 halves of `cst`).
__device__ __forceinline__ void pt_expand_plane(const uint32_t* kw, int p, int tk, int hv, uint32_t cst, uint8_t* tile) {
  constexpr int KB = 3;
  const int tl = tk >> 4, g8 = tk & 7, rr = (tk >> 3) & 1;
  uint32_t w[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) w[c] = kw[((tl * KB + p) * 32 + 4 * g8 + c) * 2 + rr];
#pragma unroll
  for (int mm = 0; mm < 4; ++mm) {
    const int m = 4 * hv + mm;  // page bit m (and m + 16) holds coordinates 8 m + 2 c (+ 1)
    uint32_t u4[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) u4[c] = (~(w[c] << (15 - m)) & 0x80008000u) | cst;
    *reinterpret_cast<uint4*>(tile + sw128_offset(tk, 8 * m)) = make_uint4(u4[0], u4[1], u4[2], u4[3]);
  }
}

// The dequantised values of a page as the B tile of P.V: V^T[j][token] = s_g (code - offset) (f16), row j = tk,
// tokens 32 hv .. 32 hv + 31 (4 chunks of 8).
template <int VB>
__device__ __forceinline__ void pt_expand_values(const uint8_t* page, const PageLayout& pl, int tk, int hv,
                                                 __half2 voff2, uint8_t* tile) {
  constexpr int D = 128;
  const int j = tk;
  const int mt = j >> 4, g8 = j & 7, rowhi = (j >> 3) & 1, grp = j >> 5;
  const uint32_t* vw = reinterpret_cast<const uint32_t*>(page + pl.vbits_off);
  const uint32_t* vsc = reinterpret_cast<const uint32_t*>(page + pl.vscale_off);  // [token pair][group] f16x2
#pragma unroll
  for (int mm = 0; mm < 4; ++mm) {
    const int m = 4 * hv + mm, blk = m >> 2, kap = (m >> 1) & 1, hiT = m & 1, rr = rowhi + 2 * hiT;
    uint32_t u4[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t x;
      if (VB == 2) {
        x = code_pair_512<2>(vw[(blk * (D / 16) + mt) * 32 + 4 * g8 + c], 2 * vfield2(kap, rr));
      } else {
        x = code_pair_512<4>(vw[((blk * (D / 16) + mt) * 32 + 4 * g8 + c) * 2 + kap], 4 * vfield4(rr));
      }
      const int t0 = 8 * m + 2 * c;  // the pair (t0, t0 + 1)
      const uint32_t s2 = vsc[(t0 >> 1) * (D / 32) + grp];
      const __half2 v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&x), voff2),
                                *reinterpret_cast<const __half2*>(&s2));
      u4[c] = *reinterpret_cast<const uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(tile + sw128_offset(j, 8 * m)) = make_uint4(u4[0], u4[1], u4[2], u4[3]);
  }
}

// Issues 8 MMAs (K = 128) of an f16 A tile against an f16 B tile, both in shared memory, into TMEM column t_d
// (descriptors stepped by one add: atom 16 KB = 1024, k step 32 B = 2, in 16-byte units).
__device__ __forceinline__ void pt_mma_k128(uint32_t t_d, uint32_t a_addr, uint32_t b_addr, bool accumulate_first) {
  const uint32_t ad = umma_desc_sw128_lo(a_addr), bd = umma_desc_sw128_lo(b_addr);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t koff = (ks >> 2) * 1024u + (ks & 3) * 2u;
    umma_bf16_lo(t_d, ad + koff, bd + koff, kIdescF16M128N128, (accumulate_first || ks > 0) ? 1u : 0u);
  }
}

// The same with the A tile in TMEM at column t_a (8 columns per K = 16 step).
__device__ __forceinline__ void pt_mma_ts_k128(uint32_t t_d, uint32_t t_a, uint32_t b_addr, bool accumulate_first) {
  const uint32_t bd = umma_desc_sw128_lo(b_addr);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t koff = (ks >> 2) * 1024u + (ks & 3) * 2u;
    umma_ts_lo(t_d, t_a + 8u * ks, bd + koff, kIdescF16M128N128, (accumulate_first || ks > 0) ? 1u : 0u);
  }
}

// One page of one KV head expanded for every query tile of the launch (grid: 2 x pages, KV heads, batch
// rows; CTA 2 p + half does half `half` of page p): the packed page is copied in; half 0 expands the h and
// l planes with n_t as fp32, half 1 the QJL plane and V^T, into shared memory in the tensor cores' layout;
// the bytes go out to the workspace by bulk copies. (Halves of 80 KB of shared memory let two CTAs share
// an SM.)
template <int VB>
__global__ void __launch_bounds__(kPtWorkers, 2) k_prefill_expand(PrefillTcArgs a) {
  constexpr int D = 128, KB = 3;
  constexpr float kVoff = VB == 2 ? 513.5f : 519.5f;  // 512 + the mid-rise offset 2^(VB-1) - 1/2
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, tk = tid & 127, hv = tid >> 7;
  const int pg = blockIdx.x >> 1, half = blockIdx.x & 1, h = blockIdx.y, b = blockIdx.z;
  const PageLayout pl = page_layout(D, VB, KB);
  uint8_t* stg = sm + 2 * kPxTileBytes + 512;  // the packed page
  uint64_t* bar = reinterpret_cast<uint64_t*>(stg + 15872);
  pdl_wait();  // pages and sequence state come from earlier work on the stream
  pdl_launch();
  const int slot = a.seq_ids[b];
  if (slot < 0 || slot >= lv.max_seqs) return;
  const int L = lv.state[2 * slot], F = lv.state[2 * slot + 1];
  const int P = (L > 0 ? kPage * ((L - 1) / kPage) : 0) + F;  // packed tokens
  if (pg * kPage >= P) return;
  if (tid == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    mbar_expect_tx(bar, pl.bytes);
    bulk_g2s(stg, pt_page(lv, slot, h, pg), pl.bytes, bar);
  }
  // thread 0 polls; the barrier makes the landed page visible to every thread
  if (!__syncthreads_and(tid == 0 ? mbar_wait(bar, 0) : true)) {
    if (tid == 0) {  // the copy may still land: wait again (bounded) before the CTA leaves its shared memory
      set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
      mbar_wait(bar, 0);
    }
    return;
  }
  const uint32_t* kw = reinterpret_cast<const uint32_t*>(stg + pl.kbits_off);
  const uint32_t nw = reinterpret_cast<const uint32_t*>(stg + pl.norms_off)[tk];
  if (half == 0) {
    if (hv == 0) reinterpret_cast<float*>(sm + 2 * kPxTileBytes)[tk] = __half2float(__ushort_as_half((uint16_t)(nw & 0xffffu)));
    pt_expand_plane(kw, 0, tk, hv, 0x3C003C00u, sm);                  // h: +-1
    pt_expand_plane(kw, 1, tk, hv, 0x3C003C00u, sm + kPxTileBytes);   // l: +-1
  } else {
    pt_expand_plane(kw, 2, tk, hv, (nw >> 16) * 0x00010001u, sm);     // QJL: +-gamma_t
    pt_expand_values<VB>(stg, pl, tk, hv, __floats2half2_rn(kVoff, kVoff), sm + kPxTileBytes);
  }
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // generic-proxy writes -> the bulk copy
  __syncthreads();
  if (tid == 0) {
    uint8_t* dst = a.ws + a.plan.px_off + (((size_t)b * lv.Hkv + h) * a.plan.px_pages + pg) * kPxBytes;
    bulk_s2g(dst + 2 * half * kPxTileBytes, sm, (uint32_t)kPxTileBytes);
    bulk_s2g(dst + (2 * half + 1) * kPxTileBytes, sm + kPxTileBytes, (uint32_t)kPxTileBytes);
    if (half == 0) bulk_s2g(dst + 4 * kPxTileBytes, sm + 2 * kPxTileBytes, 512);
    bulk_s2g_wait();  // written before the CTA leaves its shared memory
  }
}

// HOOK: the instantiation with the wait-timeout test hook compiled in (launched only while it is set).
template <int VB, bool HOOK>
__global__ void __launch_bounds__(kPtThreads, 1) k_prefill_tc(PrefillTcArgs a) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, h = blockIdx.y;
  const int S = a.plan.n_splits;
  const int b = blockIdx.z / S, split = blockIdx.z % S;
  float* ns = reinterpret_cast<float*>(sm + kPtTail0);  // [2][128] n_t of the pages in flight, by page parity
  float* xrow = ns + 256;                                // [4][128] row maxima / sums of the four quarters
  float* bmax = xrow + 512;                              // [16] per-warp operand maxima
  uint64_t* bars = reinterpret_cast<uint64_t*>(bmax + 16);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 8);
  auto tile_at = [sm](int i) { return sm + i * kPtTileBytes; };
  // this thread's query row (TMEM lane) and column quarter: columns 32 ch .. 32 ch + 31
  const int r = 32 * (warp & 3) + lane, ch = warp >> 2;
  const int qi = r >> 2, g = r & 3, qidx = 32 * tile + qi;
  const bool worker = tid < kPtWorkers;
  // The stream wait comes only before the first page copy: the sequence state, the queries and the tables
  // come from work before the expansion kernel, which was complete when that kernel passed its own wait
  // (and started this one). The setup below overlaps the expansion's last CTAs.
  const int slot = a.seq_ids[b], nq = a.n_q[b];
  const bool slot_ok = slot >= 0 && slot < lv.max_seqs;
  int P = 0, L = 0;
  if (slot_ok) {
    L = lv.state[2 * slot];
    const int F = lv.state[2 * slot + 1];
    P = (L > 0 ? kPage * ((L - 1) / kPage) : 0) + F;
  }
  // packed tokens that query i sees (causal: every position up to its own, L - (nq - 1 - i) tokens)
  auto vis = [&](int i) { return (i < nq && i < a.qpr) ? min(P, max(0, L - (nq - 1 - i))) : 0; };
  const int i_last = min(32 * tile + 31, min(nq, a.qpr) - 1);
  int npg_tile = i_last >= 32 * tile ? (vis(i_last) + kPage - 1) / kPage : 0;
  if (npg_tile > a.plan.px_pages) {  // a max_ctx_hint below the row's length: the pages past it were not expanded
    if (tid == 0 && split == 0) set_status(lv.status, TQ_DEV_ERR_SPLITS);
    npg_tile = a.plan.px_pages;
  }
  const int pps = (npg_tile + S - 1) / S;
  const int pg0 = min(npg_tile, split * pps), pg1 = min(npg_tile, pg0 + pps), n = pg1 - pg0;
  const int vis_r = vis(qidx);
  // pages below this warp's smallest causal extent need no mask
  const int vis_w = __reduce_min_sync(0xffffffffu, (unsigned)vis_r);
  const bool row_out = worker && qidx < a.qpr;  // a virtual row of the launch (padding rows get an empty partial)
  float* part = row_out ? reinterpret_cast<float*>(a.ws + a.plan.part_off +
                                                   ((((size_t)b * a.qpr + qidx) * lv.Hkv + h) * S + split) *
                                                       a.plan.part_stride)
                        : nullptr;
  if (n == 0) {  // nothing visible in this split: empty partials (m = -inf, l = 0, o = 0)
    if (row_out) {
      for (int j = 32 * ch; j < 32 * ch + 32; ++j) part[2 * kMaxG + g * D + j] = 0.f;
      if (ch == 0) {
        part[g] = -INFINITY;
        part[kMaxG + g] = 0.f;
      }
    }
    return;
  }
  // this (row, KV head)'s expanded pages: page pg0 + k of the split at px(k)
  const uint8_t* px0 = a.ws + a.plan.px_off + ((size_t)b * lv.Hkv + h) * a.plan.px_pages * kPxBytes;
  auto px = [&](int k) { return px0 + (size_t)(pg0 + k) * kPxBytes; };
  // the wait-timeout test hook: a page whose h / l tiles are never copied (nor their bytes expected), so the
  // wait for them gives up after a few polls
  const int fpage = HOOK && (blockIdx.x | blockIdx.y | blockIdx.z) == 0 ? a.fault_page : -1;
  auto skip_copy = [fpage](int k) { return HOOK && k == fpage; };
  auto page_polls = [fpage, &a](int k) { return HOOK && k == fpage ? a.fault_polls : kWaitPolls; };

  // ---- setup: barriers, TMEM (512 columns), the S table for the projection ----
  if (tid == kPtIssuer) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    mbar_expect_tx(&bars[kBarTab], 2u * D * D);
    bulk_g2s(tile_at(2), lv.S_sw, 2u * D * D, &bars[kBarTab]);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(tslot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  // ---- query rows: q_rot = Pi q (warp-per-row FWHT), bf16 hi / lo for the projection, fp32 copy ----
  // [128][128] fp32 q_rot (tiles 4-5 until the first page); column j of row r at j ^ (r mod 32), so that the
  // row-per-thread reads of the A tiles meet 32 banks
  float* qr = reinterpret_cast<float*>(tile_at(4));
  const float rs = rsqrtf((float)D);
  float amax = 0.f;
  constexpr int kRowStep = kPtWorkers / 32, kWarpRows = 128 / kRowStep;  // warp w: rows w, w + 16, ...
  uint16_t qraw[kWarpRows][4];  // every row's loads in flight before the first row's transform
  float dsg[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) dsg[e] = worker ? lv.D[4 * lane + e] : 0.f;
#pragma unroll
  for (int u = 0; u < kWarpRows; ++u) {
    const int rr = warp + u * kRowStep, i = 32 * tile + (rr >> 2), gg = rr & 3;
    const bool live = worker && i < nq && i < a.qpr && slot_ok;
    const uint16_t* src = a.q + (((size_t)b * a.qpr + i) * lv.Hq + h * kMaxG + gg) * D + 4 * lane;
#pragma unroll
    for (int e = 0; e < 4; ++e) qraw[u][e] = live ? src[e] : (uint16_t)0;
  }
#pragma unroll
  for (int u = 0; u < kWarpRows && worker; ++u) {
    const int rr = warp + u * kRowStep;
    float x[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = bf16_to_f32(qraw[u][e]) * dsg[e];
    warp_fwht<4>(x, lane);
    uint32_t hb[2], lb[2];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[e] *= rs;
      qr[rr * D + ((4 * lane + e) ^ (rr & 31))] = x[e];
      amax = fmaxf(amax, fabsf(x[e]));
    }
#pragma unroll
    for (int e2 = 0; e2 < 2; ++e2) {
      const __nv_bfloat162 hi = __floats2bfloat162_rn(x[2 * e2], x[2 * e2 + 1]);
      const float2 hf = __bfloat1622float2(hi);
      const __nv_bfloat162 lo = __floats2bfloat162_rn(x[2 * e2] - hf.x, x[2 * e2 + 1] - hf.y);
      hb[e2] = *reinterpret_cast<const uint32_t*>(&hi);
      lb[e2] = *reinterpret_cast<const uint32_t*>(&lo);
    }
    *reinterpret_cast<uint2*>(tile_at(0) + sw128_offset(rr, 4 * lane)) = make_uint2(hb[0], hb[1]);
    *reinterpret_cast<uint2*>(tile_at(1) + sw128_offset(rr, 4 * lane)) = make_uint2(lb[0], lb[1]);
  }
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot, t_s = tmem + kPtTmS, t_o = tmem + kPtTmO, t_a = tmem + kPtTmA;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  // per barrier: the parity of the next phase to wait for (bit i of par) and the phases armed (a copy or an
  // MMA batch that completes it) but not seen complete (2 bits i of pend), for the drain after a wait that
  // gave up. Every thread keeps them alike for the barriers that all threads wait for; the copy barriers
  // (kBarA, kBarB) only the issuing thread waits for and counts, and that thread runs the drain. Armed now:
  // the S table.
  uint32_t par = 0u, pend = 1u << (2 * kBarTab);
  bool iss_ok = true;  // the issuing thread's own waits all succeeded
  auto arm = [&](int i) { pend += 1u << (2 * i); };
  // A wait of the issuing thread alone (the copies it issued); a failure reaches the others at the next
  // block wait.
  auto iss_wait = [&](int i, uint32_t polls) {
    const bool w = iss_ok && mbar_wait(&bars[i], (par >> i) & 1u, polls);
    if (w) {
      par ^= 1u << i;
      pend -= 1u << (2 * i);
    }
    iss_ok = w;
    return w;
  };
  // Waits (bounded) for the oldest armed phase not seen yet of barrier i and, if j >= 0, of barrier j. The
  // issuing thread alone polls; the others wait at the block barrier, which keeps 500 pollers off the
  // shared-memory pipe that the tensor cores read their operands through (the try_wait acquire of the
  // poller and the barrier make the completed copy or MMA results visible to every thread). Every thread
  // gets the same answer.
  auto wait_bars = [&](int i, int j) {
    bool w = true;
    if (tid == kPtIssuer) {
      w = iss_ok;
      if (w && i >= 0) w = mbar_wait(&bars[i], (par >> i) & 1u);
      if (w && j >= 0) w = mbar_wait(&bars[j], (par >> j) & 1u);
    }
    w = __syncthreads_and(w) != 0;
    if (w) {
      if (i >= 0) {
        par ^= 1u << i;
        pend -= 1u << (2 * i);
      }
      if (j >= 0) {
        par ^= 1u << j;
        pend -= 1u << (2 * j);
      }
    }
    return w;
  };
  // copies of page k's h and l tiles with n_t (barrier kBarA + k % 2), and of its QJL and V^T tiles (kBarB)
  auto copy_hl = [&](int k, int th, int tl) {
    if (skip_copy(k)) return;
    uint64_t* bar = &bars[kBarA + (k & 1)];
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    mbar_expect_tx(bar, 2u * kPtTileBytes + 512u);
    bulk_g2s(tile_at(th), px(k), kPtTileBytes, bar);
    bulk_g2s(tile_at(tl), px(k) + kPxTileBytes, kPtTileBytes, bar);
    bulk_g2s(ns + 128 * (k & 1), px(k) + 4 * kPxTileBytes, 512u, bar);
    arm(kBarA + (k & 1));
  };
  auto copy_gv = [&](int k, int tg, int tv) {
    uint64_t* bar = &bars[kBarB];
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    mbar_expect_tx(bar, 2u * kPtTileBytes);
    bulk_g2s(tile_at(tg), px(k) + 2 * kPxTileBytes, kPtTileBytes, bar);
    bulk_g2s(tile_at(tv), px(k) + 3 * kPxTileBytes, kPtTileBytes, bar);
    arm(kBarB);
  };
  bool ok = wait_bars(kBarTab, -1);  // S table landed
  if (ok) {  // projection q_proj = S q_rot into TMEM columns [0, 128): A = q_rot hi, lo (bf16)
    if (tid == kPtIssuer) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 16; ++ks) {
        const uint32_t koff = ((ks & 7) >> 2) * 16384 + (ks & 3) * 32;
        umma_bf16(t_s, umma_desc_sw128(smem_u32(tile_at(ks < 8 ? 0 : 1)) + koff),
                  umma_desc_sw128(smem_u32(tile_at(2)) + koff), kIdescBf16M128N128, ks > 0);
      }
      umma_commit(&bars[kBarProj]);
    }
    arm(kBarProj);
    ok = wait_bars(kBarProj, -1);
  }
  pdl_wait();  // the expanded pages
  pdl_launch();
  // the projection has read tiles 0-2 (tile 3 was free): page 0's tiles land while the A tiles are built
  if (ok && tid == kPtIssuer) {
    copy_hl(0, 0, 1);
    copy_gv(0, 2, 3);
  }
  tc_fence_after();
  // operand scale lambda: the largest of |a_h q_rot|, |a_l q_rot| and |kappa q_proj| maps to [2^12, 2^13)
  const float w_h = lv.cb[kCbW + 0], w_l = lv.cb[kCbW + 1];
  const float kappa = 1.2533141373155003f / (float)D;  // sqrt(pi/2) / d
  float lam;
  {
    uint32_t qpv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) qpv[i] = 0u;
    if (ok && worker) tmem_ld32(t_s + lane_base + 32 * ch, qpv);
    float pmax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) pmax = fmaxf(pmax, fabsf(__uint_as_float(qpv[i])));
    const float wmax = warp_max(fmaxf(fmaxf(fabsf(w_h), fabsf(w_l)) * amax, kappa * pmax));
    if (lane == 0 && worker) bmax[warp] = wmax;
    __syncthreads();  // also: every projection MMA has read its operands (waited above)
    float tmax = 0.f;
#pragma unroll
    for (int w = 0; w < kPtWorkers / 32; ++w) tmax = fmaxf(tmax, bmax[w]);
    lam = tmax > 0.f ? exp2f(floorf(log2f(4096.f / tmax))) : 1.f;
    // The A tiles into TMEM, row r, coordinates 32 ch .. 32 ch + 31 = columns 16 ch .. 16 ch + 15 of each:
    // A_qp = lambda kappa q_proj; A_hi / A_lo = f16 hi / remainder of lambda a_h q_rot; A_l = lambda a_l q_rot
    uint32_t u[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const __half2 hv2 = __floats2half2_rn(lam * kappa * __uint_as_float(qpv[2 * i]),
                                            lam * kappa * __uint_as_float(qpv[2 * i + 1]));
      u[i] = *reinterpret_cast<const uint32_t*>(&hv2);
    }
    if (ok && worker) tmem_st16(t_a + 192 + lane_base + 16 * ch, u);
  }
  {
    uint32_t hi16[16], lo16[16], l16[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int j = (32 * ch + 2 * i) & (D - 1);  // (the issuing warp's values are not stored)
      const float q0 = qr[r * D + (j ^ (r & 31))], q1 = qr[r * D + ((j + 1) ^ (r & 31))];
      const float x0 = lam * w_h * q0, x1 = lam * w_h * q1;
      const __half2 hi = __floats2half2_rn(x0, x1);
      const float2 hf = __half22float2(hi);
      const __half2 lo = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
      const __half2 lp = __floats2half2_rn(lam * w_l * q0, lam * w_l * q1);
      hi16[i] = *reinterpret_cast<const uint32_t*>(&hi);
      lo16[i] = *reinterpret_cast<const uint32_t*>(&lo);
      l16[i] = *reinterpret_cast<const uint32_t*>(&lp);
    }
    if (ok && worker) {
      tmem_st16(t_a + 0 + lane_base + 16 * ch, hi16);
      tmem_st16(t_a + 64 + lane_base + 16 * ch, lo16);
      tmem_st16(t_a + 128 + lane_base + 16 * ch, l16);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
  }
  const float logit = a.scale * 1.4426950408889634f / lam;  // S n_t logit = score in log2 units
  tc_fence_before();
  __syncthreads();  // the A tiles are in TMEM; every qr read is done, so all six operand tiles are free
  // Page pipeline. Page k's h, l, QJL and V^T tiles sit in tiles sH, sL, sG, sV; f1 and f2 are free. The
  // issuing thread copies the expanded tiles in and issues the MMAs; the workers run the softmax. Page k's
  // score MMAs run in two parts: the h and l planes (24 MMAs) as soon as page k - 1's softmax has read S,
  // the QJL plane (8) right after page k - 1's P.V MMAs. The MMAs of one thread run in issue order, so S of
  // page k is complete only after the P.V MMAs of page k - 1. In iteration k:
  //   - once the previous P.V MMAs are done (f1, f2 free), the issuer copies page k + 1's h and l tiles
  //     and n_t into f1, f2; everyone waits for page k's scores;
  //   - the workers read S, exchange row maxima, then finish the softmax, with P (f16) over the h tile;
  //     meanwhile the issuer copies page k + 1's QJL and V^T tiles into the l and QJL tiles of page k
  //     (its scores are done) and issues page k + 1's h and l MMAs once their tiles have landed;
  //   - the issuer issues the P.V MMAs of page k, then page k + 1's QJL MMAs once its QJL tile has landed.
  // The tiles then rotate: page k + 1 has h = f1, l = f2, QJL = sL, V = sG, and sH, sV (P and V of page k)
  // are free once the P.V MMAs have read them. The rotation has period 4 (page 0: h, l, QJL, V = tiles 0-3,
  // f1, f2 = 4, 5); tile_of reads role r's tile for page k from a table of 4-bit fields, one per k % 4.
  constexpr uint32_t kRoleH = 0x4040, kRoleL = 0x2351, kRoleG = 0x3512, kRoleV = 0x5123, kRoleF1 = 0x0404,
                     kRoleF2 = 0x1235;
  auto tile_of = [](uint32_t role, int k) { return (int)((role >> (4 * (k & 3))) & 7u); };
  // S = A_hi H + A_lo H + A_l L (issue_hl, committed to kBarHL) + A_qp G (committed to kBarS)
  auto issue_hl = [&](int th, int tl) {
    tc_fence_after();
    pt_mma_ts_k128(t_s, t_a + 0, smem_u32(tile_at(th)), false);
    pt_mma_ts_k128(t_s, t_a + 64, smem_u32(tile_at(th)), true);
    pt_mma_ts_k128(t_s, t_a + 128, smem_u32(tile_at(tl)), true);
    umma_commit(&bars[kBarHL]);
    arm(kBarHL);
  };
  // page 0's QJL MMAs (committed to kBarS)
  auto issue_g = [&](int tg) {
    tc_fence_after();
    pt_mma_ts_k128(t_s, t_a + 192, smem_u32(tile_at(tg)), true);
    umma_commit(&bars[kBarS]);
    arm(kBarS);
  };
  if (ok && tid == kPtIssuer) {  // page 1's h and l tiles (the A tiles have read qr); page 0's score MMAs
    if (n > 1) copy_hl(1, 4, 5);
    if (iss_wait(kBarA, page_polls(0))) issue_hl(0, 1);
    if (iss_wait(kBarB, kWaitPolls)) issue_g(2);
  }
  if (tid != kPtIssuer && ok) {  // (the issuer counts them only if issued)
    arm(kBarHL);
    arm(kBarS);
  }
  float m_used = -INFINITY, l_loc = 0.f;
  for (int k = 0; k < n && ok; ++k) {
    const int pg = pg0 + k, st = k & 1;
    const bool more = k + 1 < n;
    const int sH = tile_of(kRoleH, k), sL = tile_of(kRoleL, k), sG = tile_of(kRoleG, k), sV = tile_of(kRoleV, k);
    const int f1 = tile_of(kRoleF1, k), f2 = tile_of(kRoleF2, k);
    // the previous P.V MMAs are done: f1, f2 are free (page 1's h and l tiles were copied before the loop).
    // Every P.V batch is waited for here, the last page's predecessor too: a parity wait cannot tell a
    // phase from the one two later, so no two phases of a barrier may complete unseen.
    if (tid == kPtIssuer && k > 0 && iss_wait(kBarO, kWaitPolls) && more) copy_hl(k + 1, f1, f2);
    // ---- softmax of row r over tokens 32 ch .. 32 ch + 31 of page k ----
    ok = wait_bars(kBarS, kBarHL);  // page k's scores (and so the previous P.V MMAs) are complete
    if (!ok) break;
    tc_fence_after();
    uint32_t sv[32];
    float mx = -INFINITY;
    if (worker) {
      tmem_ld32(t_s + lane_base + 32 * ch, sv);
      const bool full = pg * kPage + kPage <= vis_w;  // every token of the page is visible to the whole warp
      const float* nsk = ns + 128 * st;
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4) {
        const float4 f = *reinterpret_cast<const float4*>(nsk + 32 * ch + 4 * i4);
        const float fv[4] = {f.x * logit, f.y * logit, f.z * logit, f.w * logit};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = 4 * i4 + e, t = 32 * ch + i;
          float s = __uint_as_float(sv[i]) * fv[e];
          if (!full && pg * kPage + t >= vis_r) s = -INFINITY;
          sv[i] = __float_as_uint(s);
          mx = fmaxf(mx, s);
        }
      }
      xrow[128 * ch + r] = mx;
    }
    tc_fence_before();
    __syncthreads();  // S is read: the next page's h and l MMAs may overwrite it
    if (tid == kPtIssuer && more) {
      copy_gv(k + 1, sL, sG);  // page k's scores are done: its l and QJL tiles are free
      if (iss_wait(kBarA + ((k + 1) & 1), page_polls(k + 1))) issue_hl(f1, f2);
    }
    if (tid != kPtIssuer && more) arm(kBarHL);
    if (worker) {
#pragma unroll
      for (int q = 1; q < kPtQ; ++q) mx = fmaxf(mx, xrow[128 * ((ch + q) % kPtQ) + r]);
      // the row maximum grew by more than 2^8: move to the new maximum (O and l scaled by alpha). The TMEM
      // loads and stores are warp-wide, so a warp rescales when any of its rows needs it (alpha = 1 for the
      // rest). The previous P.V MMAs are done (waited above).
      const bool grow = mx > m_used + 8.f;
      const float alpha = !grow ? 1.f : (m_used == -INFINITY ? 0.f : pt_ex2(m_used - mx));
      if (__any_sync(0xffffffffu, grow && k > 0)) {
        uint32_t ov[32];
        tmem_ld32(t_o + lane_base + 32 * ch, ov);
#pragma unroll
        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
        tmem_st32(t_o + lane_base + 32 * ch, ov);
      }
      if (grow) {
        l_loc *= alpha;
        m_used = mx;
      }
      const float mref = m_used == -INFINITY ? 0.f : m_used;  // every s is -inf while nothing is visible
#pragma unroll
      for (int mm = 0; mm < 4; ++mm) {
        uint32_t u4[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int i = 8 * mm + 2 * c;
          const float p0 = pt_ex2(__uint_as_float(sv[i]) - mref), p1 = pt_ex2(__uint_as_float(sv[i + 1]) - mref);
          l_loc += p0 + p1;
          const __half2 ph = __floats2half2_rn(p0, p1);
          u4[c] = *reinterpret_cast<const uint32_t*>(&ph);
        }
        *reinterpret_cast<uint4*>(tile_at(sH) + sw128_offset(r, 32 * ch + 8 * mm)) =
            make_uint4(u4[0], u4[1], u4[2], u4[3]);
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    if (tid == kPtIssuer && iss_ok) {  // O += P V: A = P [rows x tokens] (over the h tile), B = V^T
      tc_fence_after();
      pt_mma_k128(t_o, smem_u32(tile_at(sH)), smem_u32(tile_at(sV)), k > 0);
      umma_commit(&bars[kBarO]);  // (also covers the next page's h and l MMAs issued before)
      arm(kBarO);
      if (more && iss_wait(kBarB, kWaitPolls)) issue_g(sL);  // page k + 1's QJL tile sits in page k's l tile
    }
    if (tid != kPtIssuer && more) arm(kBarS);
  }
  // the last P.V batch (the issuing thread's wait, which the others learn of at the block barrier)
  if (tid == kPtIssuer && ok && ((pend >> (2 * kBarO)) & 3u)) iss_wait(kBarO, kWaitPolls);
  ok = __syncthreads_and(tid == kPtIssuer ? ok && iss_ok : ok) != 0;
  tc_fence_after();
  // ---- the partial of row r: m (log2 units), l, o (rotated basis, relative to m) ----
  __syncthreads();  // every thread has read the row maxima above
  if (worker) xrow[128 * ch + r] = l_loc;
  __syncthreads();
  float l_row = 0.f;
#pragma unroll
  for (int q = 0; q < kPtQ; ++q) l_row += worker ? xrow[128 * q + r] : 0.f;
  const bool has = ok && m_used != -INFINITY;  // this row saw a token
  if (ok) {
    // O through shared memory (tiles 0-2 are free: every copy and MMA was seen complete), rows padded to
    // 132 floats so that eight rows' float4 stores meet eight bank quads; then warp w stores rows w, w + 16,
    // ..., a whole 512-byte row per store
    float* ost = reinterpret_cast<float*>(sm);
    if (worker) {
      uint32_t ov[32];
      tmem_ld32(t_o + lane_base + 32 * ch, ov);
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4)
        *reinterpret_cast<float4*>(ost + r * 132 + 32 * ch + 4 * i4) =
            has ? make_float4(__uint_as_float(ov[4 * i4]), __uint_as_float(ov[4 * i4 + 1]),
                              __uint_as_float(ov[4 * i4 + 2]), __uint_as_float(ov[4 * i4 + 3]))
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    for (int rr = warp; rr < 128 && worker; rr += kPtWorkers / 32) {
      const int qx = 32 * tile + (rr >> 2);
      if (qx >= a.qpr) continue;
      float* pr = reinterpret_cast<float*>(a.ws + a.plan.part_off +
                                           ((((size_t)b * a.qpr + qx) * lv.Hkv + h) * S + split) *
                                               a.plan.part_stride);
      *reinterpret_cast<float4*>(pr + 2 * kMaxG + (rr & 3) * D + 4 * lane) =
          *reinterpret_cast<const float4*>(ost + rr * 132 + 4 * lane);
    }
  } else if (row_out) {  // a wait gave up (copies may still land in shared memory): an empty O
#pragma unroll
    for (int i4 = 0; i4 < 8; ++i4)
      *reinterpret_cast<float4*>(part + 2 * kMaxG + g * D + 32 * ch + 4 * i4) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (row_out && ch == 0) {
    part[g] = has ? m_used : -INFINITY;
    part[kMaxG + g] = has ? l_row : 0.f;
  }
  if (!ok && tid == kPtIssuer) {
    // a wait gave up: nothing more is issued; wait (bounded) for every armed phase not seen complete - the
    // MMA batches before TMEM is freed, the copies before the CTA leaves its shared memory
    set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
    for (int i = 0; i < kNumBars; ++i)
      for (uint32_t c = 0, ph = (par >> i) & 1u; c < ((pend >> (2 * i)) & 3u); ++c, ph ^= 1u) mbar_wait(&bars[i], ph);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem) : "memory");
}

// The third launch: for each (query, KV head), the exact ring split and the combine. The ring tokens the
// query sees (positions P .. its own) are bf16 K and V rows of the ring, attended exactly in fp32 in the
// original basis (TurboQuant vLLM guide, §五.1: the recent tokens kept unquantised; §三: the hybrid decode
// merges both parts). The history partials of the tile kernel's splits (m in log2 units, l, o in the rotated
// basis relative to m) merge by log-sum-exp, o goes back through Pi^T = diag(D) H / sqrt(d), and the two
// parts merge exactly. One CTA per (query, KV head): warp g ends with query head g of the group, lane l with
// coordinates 4 l .. 4 l + 3. Queries past n_q, and rows with an invalid sequence id, get zeros.
__global__ void __launch_bounds__(32 * kMaxG, 4) k_prefill_ring(PrefillTcArgs a, float* out) {
  constexpr int D = 128;
  const LayerView& lv = a.lv;
  const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  __shared__ float qs[kMaxG][D];
  pdl_wait();  // the partials of the tile kernel (and the state, ring and queries of earlier work)
  pdl_launch();
  // the history partials first: their loads depend on nothing else (every row < q_per_row has them)
  const int S = a.plan.n_splits;
  const size_t stride = a.plan.part_stride / sizeof(float);
  const float* base = reinterpret_cast<const float*>(a.ws + a.plan.part_off +
                                                     (((size_t)b * a.qpr + i) * lv.Hkv + h) * S *
                                                         a.plan.part_stride);
  float ms[2], ls[2];  // splits lane and lane + 32 (S <= 64)
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int sp = lane + 32 * u;
    ms[u] = sp < S ? __ldcg(base + sp * stride + g) : -INFINITY;
    ls[u] = sp < S ? __ldcg(base + sp * stride + kMaxG + g) : 0.f;
  }
  constexpr int kPre = 8;  // the first splits' o rows, in flight with the loads above
  float4 opre[kPre];
#pragma unroll
  for (int u = 0; u < kPre; ++u)
    opre[u] = u < S ? __ldcg(reinterpret_cast<const float4*>(base + u * stride + 2 * kMaxG + g * D + 4 * lane))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
  float* dst = out + (((size_t)b * a.qpr + i) * lv.Hq + h * kMaxG + g) * D + 4 * lane;
  const int slot = a.seq_ids[b], nq = a.n_q[b];
  if (i >= nq || slot < 0 || slot >= lv.max_seqs) {
    *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int L = lv.state[2 * slot], F = lv.state[2 * slot + 1];
  const int P = (L > 0 ? kPage * ((L - 1) / kPage) : 0) + F;  // packed tokens read through their codes
  const int n = max(0, L - (nq - 1 - i)) - P;                  // ring tokens this query sees (<= 128)
  // ---- ring split (n is the same in the whole CTA). Thread t scores ring token t for the four heads;
  // warp w takes tokens 32 w .. 32 w + 31 of P.V for the four heads over this lane's coordinates, and
  // warp g then sums head g's four parts. ----
  float m_r = -INFINITY, l_r = 0.f, o_r[4] = {0.f, 0.f, 0.f, 0.f};
  if (n > 0) {
    __shared__ float ps[kMaxG][kPage];      // p_t of each head
    __shared__ float red[2][kMaxG][kMaxG];  // per-warp maxima, then sums, of each head
    __shared__ float4 ored[kMaxG][kMaxG][32];  // [warp][head][lane] parts of P.V
    const int t = threadIdx.x;
    {
      const uint16_t* qrow = a.q + (((size_t)b * a.qpr + i) * lv.Hq + h * kMaxG + g) * D + 4 * lane;
      const uint2 qw = *reinterpret_cast<const uint2*>(qrow);
      qs[g][4 * lane + 0] = __uint_as_float(qw.x << 16);
      qs[g][4 * lane + 1] = __uint_as_float(qw.x & 0xffff0000u);
      qs[g][4 * lane + 2] = __uint_as_float(qw.y << 16);
      qs[g][4 * lane + 3] = __uint_as_float(qw.y & 0xffff0000u);
    }
    __syncthreads();
    const uint16_t* rk = lv.ring + ((size_t)slot * lv.Hkv + h) * 2 * kPage * D + (size_t)F * D;
    const uint16_t* rv = rk + (size_t)kPage * D;
    const float s2 = a.scale * 1.4426950408889634f;  // scores in log2 units
    float sc[kMaxG] = {0.f, 0.f, 0.f, 0.f};
    if (t < n) {
      const uint4* krow = reinterpret_cast<const uint4*>(rk + (size_t)t * D);
      constexpr int KH = D / 16;  // the row in two halves of 8 chunks: half the registers in flight
#pragma unroll
      for (int hk = 0; hk < 2; ++hk) {
        uint4 kw[KH];
#pragma unroll
        for (int u = 0; u < KH; ++u) kw[u] = krow[KH * hk + u];
#pragma unroll
        for (int u = 0; u < KH; ++u) {
          const int c = KH * hk + u;
          const float k8[8] = {__uint_as_float(kw[u].x << 16), __uint_as_float(kw[u].x & 0xffff0000u),
                               __uint_as_float(kw[u].y << 16), __uint_as_float(kw[u].y & 0xffff0000u),
                               __uint_as_float(kw[u].z << 16), __uint_as_float(kw[u].z & 0xffff0000u),
                               __uint_as_float(kw[u].w << 16), __uint_as_float(kw[u].w & 0xffff0000u)};
#pragma unroll
          for (int gg = 0; gg < kMaxG; ++gg) {
            const float4 q0 = *reinterpret_cast<const float4*>(&qs[gg][8 * c]);
            const float4 q1 = *reinterpret_cast<const float4*>(&qs[gg][8 * c + 4]);
            float acc = sc[gg];
            acc = fmaf(q0.x, k8[0], acc);
            acc = fmaf(q0.y, k8[1], acc);
            acc = fmaf(q0.z, k8[2], acc);
            acc = fmaf(q0.w, k8[3], acc);
            acc = fmaf(q1.x, k8[4], acc);
            acc = fmaf(q1.y, k8[5], acc);
            acc = fmaf(q1.z, k8[6], acc);
            acc = fmaf(q1.w, k8[7], acc);
            sc[gg] = acc;
          }
        }
      }
    }
#pragma unroll
    for (int gg = 0; gg < kMaxG; ++gg) {
      sc[gg] = t < n ? sc[gg] * s2 : -INFINITY;
      const float wm = warp_max(sc[gg]);
      if (lane == 0) red[0][g][gg] = wm;
    }
    __syncthreads();
    float mh[kMaxG];
#pragma unroll
    for (int gg = 0; gg < kMaxG; ++gg) {
      mh[gg] = fmaxf(fmaxf(red[0][0][gg], red[0][1][gg]), fmaxf(red[0][2][gg], red[0][3][gg]));
      const float p = t < n ? exp2f(sc[gg] - mh[gg]) : 0.f;
      ps[gg][t] = p;
      const float ws = warp_sum(p);
      if (lane == 0) red[1][g][gg] = ws;
    }
    __syncthreads();
    m_r = mh[g];
    l_r = (red[1][0][g] + red[1][1][g]) + (red[1][2][g] + red[1][3][g]);
    float4 op[kMaxG];
#pragma unroll
    for (int gg = 0; gg < kMaxG; ++gg) op[gg] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int t1 = min(n, 32 * g + 32);  // this warp's tokens 32 g .. t1 - 1
#pragma unroll 16
    for (int tt = 32 * g; tt < t1; ++tt) {
      const uint2 vw = *reinterpret_cast<const uint2*>(rv + (size_t)tt * D + 4 * lane);
      const float v0 = __uint_as_float(vw.x << 16), v1 = __uint_as_float(vw.x & 0xffff0000u);
      const float v2 = __uint_as_float(vw.y << 16), v3 = __uint_as_float(vw.y & 0xffff0000u);
#pragma unroll
      for (int gg = 0; gg < kMaxG; ++gg) {
        const float p = ps[gg][tt];
        op[gg].x = fmaf(p, v0, op[gg].x);
        op[gg].y = fmaf(p, v1, op[gg].y);
        op[gg].z = fmaf(p, v2, op[gg].z);
        op[gg].w = fmaf(p, v3, op[gg].w);
      }
    }
#pragma unroll
    for (int gg = 0; gg < kMaxG; ++gg) ored[g][gg][lane] = op[gg];
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kMaxG; ++w) {
      const float4 v = ored[w][g][lane];
      o_r[0] += v.x;
      o_r[1] += v.y;
      o_r[2] += v.z;
      o_r[3] += v.w;
    }
  }
  // ---- the history splits: weights 2^(m_s - m) with m their maximum ----
  const float m = warp_max(fmaxf(ms[0], ms[1]));
  float wl = 0.f;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    ms[u] = ms[u] == -INFINITY ? 0.f : exp2f(ms[u] - m);  // the split's weight
    wl = fmaf(ms[u], ls[u], wl);
  }
  const float l = warp_sum(wl);
  float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const float w = __shfl_sync(0xffffffffu, ms[0], u);  // 0 past S
    o[0] = fmaf(w, opre[u].x, o[0]);
    o[1] = fmaf(w, opre[u].y, o[1]);
    o[2] = fmaf(w, opre[u].z, o[2]);
    o[3] = fmaf(w, opre[u].w, o[3]);
  }
#pragma unroll 8
  for (int sp = kPre; sp < S; ++sp) {
    const float w = __shfl_sync(0xffffffffu, sp < 32 ? ms[0] : ms[1], sp & 31);
    const float4 v = __ldcg(reinterpret_cast<const float4*>(base + sp * stride + 2 * kMaxG + g * D + 4 * lane));
    o[0] = fmaf(w, v.x, o[0]);
    o[1] = fmaf(w, v.y, o[1]);
    o[2] = fmaf(w, v.z, o[2]);
    o[3] = fmaf(w, v.w, o[3]);
  }
  // Pi^T o = D * (H o) / sqrt(d), then the exact merge with the ring
  warp_fwht<4>(o, lane);
  const float rs = rsqrtf((float)D);
  const float mm = fmaxf(m, m_r);
  const float fh = m == -INFINITY ? 0.f : exp2f(m - mm), fr = m_r == -INFINITY ? 0.f : exp2f(m_r - mm);
  const float den = fh * l + fr * l_r, inv = den > 0.f ? 1.f / den : 0.f;
  float r[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) r[e] = (fh * o[e] * rs * lv.D[4 * lane + e] + fr * o_r[e]) * inv;
  *reinterpret_cast<float4*>(dst) = make_float4(r[0], r[1], r[2], r[3]);
}

}  // namespace

bool prefill_tc_eligible(const tq_ctx* ctx) {
  const tq_config& c = ctx->cfg;
  return c.head_dim == 128 && c.key_bits == 3 && c.n_q_heads == kMaxG * c.n_kv_heads;
}

int prefill_tc_splits(const tq_ctx* ctx, int batch, int q_per_row, int max_ctx_hint) {
  const int hint = (max_ctx_hint <= 0 || max_ctx_hint > ctx->cfg.max_ctx) ? ctx->cfg.max_ctx : max_ctx_hint;
  const int max_pages = std::max(1, (hint + kPage - 1) / kPage);
  const long long tiles = (long long)(q_per_row + 31) / 32 * ctx->cfg.n_kv_heads * batch;
  const long long sms = ctx->sm_count > 0 ? ctx->sm_count : 152;
  // The CTAs run in waves of one per SM, each over ceil(pages / S) pages after a fixed cost (the S table,
  // the query rows and their projection, the pipeline's first copies, the partial's write: about 17 us,
  // six pages' time, measured). The split count with the earliest end of the last wave wins (the smaller
  // on a tie): 128 tiles of 256 pages on 152 SMs take 7 splits, six waves of 37 pages (741 us per launch),
  // against one wave of 256 pages on 128 SMs (758 us).
  constexpr long long kSetupPages = 6;
  int best = 1;
  long long best_t = -1;
  for (int S = 1; S <= std::min(max_pages, 64); ++S) {
    const long long waves = (tiles * S + sms - 1) / sms, t = waves * ((max_pages + S - 1) / S + kSetupPages);
    if (best_t < 0 || t < best_t) {
      best = S;
      best_t = t;
    }
  }
  return best;
}

template <int VB>
cudaError_t launch_prefill_expand_k(const PrefillTcArgs& a, int batch, cudaStream_t s) {
  constexpr size_t smem = prefill_expand_smem();
  static bool attr = false;  // set once, outside any stream capture that follows
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_prefill_expand<VB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(k_prefill_expand<VB>, dim3(2 * a.plan.px_pages, a.lv.Hkv, batch), dim3(kPtWorkers), smem, s, a);
}

template <int VB, bool HOOK>
cudaError_t launch_prefill_tc_k(const PrefillTcArgs& a, dim3 grid, size_t smem, cudaStream_t s) {
  static bool attr = false;  // set once, outside any stream capture that follows
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_prefill_tc<VB, HOOK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(k_prefill_tc<VB, HOOK>, grid, dim3(kPtThreads), smem, s, a);
}

cudaError_t launch_prefill_tc(const tq_ctx* ctx, int layer, const void* q, const int32_t* seq_ids, const int32_t* n_q,
                              int batch, int q_per_row, float scale, void* ws, const DecodePlan& plan, float* out,
                              cudaStream_t s) {
  PrefillTcArgs a;
  a.lv = layer_view(ctx, layer);
  a.q = static_cast<const uint16_t*>(q);
  a.seq_ids = seq_ids;
  a.n_q = n_q;
  a.qpr = q_per_row;
  a.scale = scale;
  a.ws = static_cast<uint8_t*>(ws);
  a.plan = plan;
  a.fault_page = g_pfault_page.load();
  a.fault_polls = (uint32_t)g_pfault_polls.load();
  const dim3 grid((q_per_row + 31) / 32, a.lv.Hkv, batch * plan.n_splits);
  const size_t smem = prefill_tc_smem();
  // every page of every row, expanded once for all query tiles
  cudaError_t e = a.lv.vb == 2 ? launch_prefill_expand_k<2>(a, batch, s) : launch_prefill_expand_k<4>(a, batch, s);
  if (e != cudaSuccess) return e;
  const bool hook = a.fault_page >= 0;
  e = a.lv.vb == 2 ? (hook ? launch_prefill_tc_k<2, true>(a, grid, smem, s) : launch_prefill_tc_k<2, false>(a, grid, smem, s))
                   : (hook ? launch_prefill_tc_k<4, true>(a, grid, smem, s) : launch_prefill_tc_k<4, false>(a, grid, smem, s));
  if (e != cudaSuccess) return e;
  // the ring split and the combine of every (query, KV head)
  return launch_pdl(k_prefill_ring, dim3(q_per_row, a.lv.Hkv, batch), dim3(32 * kMaxG), 0, s, a, out);
}

}  // namespace tq

extern "C" tq_status tq_debug_prefill_wait_fault(int page, int polls) {
  if (page < -1) return tq::set_error(TQ_ERR_INVALID_ARG, "page must be -1 (off) or >= 0");
  if (page >= 0 && (polls < 1 || polls > (int)tq::kWaitPolls))
    return tq::set_error(TQ_ERR_INVALID_ARG, "polls must be in [1, 2^22]");
  tq::g_pfault_polls.store(page >= 0 ? polls : 0);
  tq::g_pfault_page.store(page);
  return tq::set_error(TQ_OK, "");
}
