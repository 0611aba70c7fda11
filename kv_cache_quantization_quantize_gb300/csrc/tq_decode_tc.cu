// Hybrid decode attention at head_dim 128 with 3-bit keys on the tcgen05 tensor cores ([Guide] §五.1 and
// §七: scores straight from the packed keys plus the QJL correction, values dequantised inside an online
// softmax, exact merge with the bf16 ring).
//
// The estimator is the one of tq_decode.cu:
//   s = scale * n * ( <Pi q, c[idx]> + sqrt(pi/2)/d * gamma * <S Pi q, 2 sign - 1> ),
//   c[idx] = alpha (2 b1 - 1) + beta (2 b0 - 1)  (odd-symmetric 2-bit Lloyd-Max codebook).
// What differs is where the three key bit planes meet the query:
//   - A (tokens x 384 = 3 planes x 128 coordinates) is built in TMEM as e4m3: one LOP3 per 4 elements masks
//     bit p (0..3) of every byte of a packed key word, which as an e4m3 byte is exactly 2^(p-9) or 0.
//   - B (384 x 16) is the query in shared memory: for each of the 4 heads, four e4m3 "digits" whose sum
//     represents w_plane * lambda * x_j * 2^(9-p) to about 16 bits (x = Pi q for the index planes, S Pi q
//     for the sign plane). The 16 columns are (head, digit); the MMA products are exact and accumulate in
//     fp32, so summing a head's 4 digit columns gives the plane dot products.
//   - tcgen05.mma kind::f8f6f4, M = 128 tokens, N = 16, K = 32: 8 k-steps (index planes) into one TMEM
//     accumulator and 4 (sign plane) into another, 12 MMAs per 128-token page, issued by one thread.
// Values keep the f16 mma.sync path of tq_decode.cu (code fields as f16 subnormals against P' = p s 2^(24-pos),
// mid-rise offset per page), fed with P' from shared memory.
//
// Warp roles of a split CTA (16 warps, one CTA per SM):
//   warp 0        producer: bulk copies of whole pages into a ring of stages (mbarrier complete_tx);
//   warp 1        TMEM owner and MMA issuer;
//   warps 4-7     key expanders: thread t builds row t (token t) of the page's A in TMEM;
//   warps 8-11    softmax: thread t reads token t's 32 accumulators, forms its 4 head scores, and with its
//                 warp's 32 tokens the running max, p and P' for value warp (warp - 8);
//   warps 12-15   value warps: warp 12 + w runs P.V for tokens 32w .. 32w + 31 of every page.
// Softmax warp w and value warp w share one running max per head, so no barrier spans more than a warp
// pair; the four (m, l, O) partials are merged once at the end. Pages flow through TMEM in NB buffers
// (A: 96 columns, scores: 32 columns), so expansion, MMAs, softmax and P.V of different pages overlap.
// Every wait is bounded: a wait that gives up sets an abort flag that every role polls, all roles leave
// their loops, the copies and MMAs that were issued are waited for (bounded), and the call reports
// TQ_DEV_ERR_TIMEOUT.
#include <algorithm>

#include <cuda_fp8.h>

#include "tq_decode_common.cuh"

namespace tq {
namespace {

constexpr int kTcD = 128;
constexpr int kTcThreads = 512;
constexpr int kTcNB = 4;           // TMEM page buffers (4 x 128 columns)
constexpr int kTcKSteps = 12;      // 3 planes x 4 words of 32 coordinates
constexpr int kTcPRow = 136;       // f16 per row of a P' buffer (128 tokens + 8 of padding: conflict-free loads)

template <int VB>
__host__ __device__ constexpr int tc_stages() {  // pages in flight per CTA
  return VB == 2 ? 12 : 9;
}

// Shared memory (dynamic, 1024-byte aligned base):
//   [0, 1024)       mbarriers and small state (see TcBars)
//   kTcBq           query digits, e4m3 [16 rows][384], 128-byte swizzled K-major (3 atoms of 2048 B)
//   kTcCst          per-head constants [4][4] f32: um, um cm, uq, uq cq
//   kTcAlpha        per-page rescale factors [NB][4 warps][4 heads] f32
//   kTcP            P' [NB][4 heads][kTcPRow] f16
//   kTcPrep         query prep scratch (q_rot, q_proj [4][128] f32, 32 f32)
//   kTcStage        page stages [STAGES][page bytes]; after the loop, the merge and combine scratch
constexpr uint32_t kTcBq = 1024, kTcCst = kTcBq + 6144, kTcAlpha = kTcCst + 64;
constexpr uint32_t kTcP = kTcAlpha + kTcNB * 16 * 4;
constexpr uint32_t kTcPrep = kTcP + kTcNB * 4 * kTcPRow * 2;
constexpr uint32_t kTcStage = (kTcPrep + (2 * 4 * kTcD + 32) * 4 + 127) / 128 * 128;

template <int VB>
constexpr size_t tc_smem_bytes() {
  const size_t page = (size_t)3 * kPage * kTcD / 8 + 4 * kPage + (size_t)kPage * kTcD * VB / 8 + 2 * kPage * (kTcD / 32);
  const size_t loop = kTcStage + tc_stages<VB>() * page;
  const size_t ring = ring_smem_bytes<kTcD, 1>();
  const size_t merge = kTcStage + sizeof(float) * (4 * 4 * 3 + 4 * 4 * kTcD) + sizeof(float) * (4 * 16 + 2 * 4 * 1026);
  return 1024 + std::max(std::max(loop, ring), merge);  // + alignment slack of the base
}

struct TcBars {
  uint64_t full[12], empty[12];  // page stages: copy landed / every role done with it
  uint64_t a_ready[kTcNB];       // A of the buffer written (4 expander warps)
  uint64_t mma_done[kTcNB];      // score MMAs of the buffer complete (tcgen05.commit)
  uint64_t s_free[kTcNB];        // scores of the buffer read (4 softmax warps)
  uint64_t p_ready[kTcNB][4];    // P' of value warp w written (softmax warp w)
  uint64_t p_free[kTcNB][4];     // P' of value warp w consumed (value warp w)
  uint32_t tmem;                 // TMEM base address (written by tcgen05.alloc)
  int abort;                     // a wait gave up
};
static_assert(sizeof(TcBars) <= 1024, "barrier block");

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// Bounded wait (`limit` polls) that also gives up once another role has set the abort flag.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                        uint32_t limit = kWaitPolls) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 255u) == 255u && *abort) return false;
  }
  *abort = 1;
  return false;
}

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t smem_addr) {
  return (uint64_t)((smem_addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f8f6f4: D = f32, A = B = e4m3, both K-major, N = 16, M = 128.
constexpr uint32_t kIdescE4m3M128N16 = (1u << 4) | (0u << 7) | (0u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void mma_e4m3_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(kIdescE4m3M128N16), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
}

// Byte offset of element (row n, k) of the query-digit matrix [16][384] e4m3 (128-byte swizzle, K-major:
// atoms of 16 rows x 128 bytes, 16-byte chunk c of row n stored at chunk c ^ (n & 7)).
__device__ __forceinline__ uint32_t bq_offset(int n, int k) {
  return (uint32_t)((k >> 7) * 2048 + (n >> 3) * 1024 + (n & 7) * 128 + ((((k & 127) >> 4) ^ (n & 7)) << 4) + (k & 15));
}

// Position of coordinate j (0..127) in a token's packed key words (KBITS, kbit_loc with d = 128): word
// c = (j >> 1) & 3 of the token, bit b = 2 (j >> 4) + ((j >> 3) & 1) + 16 (j & 1). In A the word becomes
// k-step 4 plane + c; its bit b lands in column 4 (b & 4 ? 1 : 0) + (b & 3) of the k-step, byte b >> 3, i.e. at
// K index 4 (4 hi + p) + (b >> 3) with p = b & 3 and hi = (b >> 2) & 1, as the e4m3 value 2^(p - 9).
__device__ __forceinline__ void coord_slot(int j, int& ks_word, int& kk, int& p) {
  const int b = 2 * (j >> 4) + ((j >> 3) & 1) + 16 * (j & 1);
  ks_word = (j >> 1) & 3;
  p = b & 3;
  kk = 4 * (4 * ((b >> 2) & 1) + p) + (b >> 3);
}

__device__ __forceinline__ uint8_t to_e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float from_e4m3(uint8_t v) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)v, __NV_E4M3);
  return __half2float(__half(h));
}

// Query prep of one (row, KV head): q_rot and q_proj (shared with tq_decode.cu), then the e4m3 digits of B
// and the per-head constants. Warp h (h < 4) builds the 4 digit rows of head h; heads >= G get zero rows.
//   index planes pl = 0, 1: X = 2 w_pl lam_m q_rot_j 2^(9-p); sign plane: X = 2 lam_q q_proj_j 2^(9-p), with
//   lam a power of two that keeps every |X| <= 448 (the largest e4m3 value) and w = alpha, beta.
//   Digits: d1 = e4m3(X), d2 = e4m3(X - d1), ... (4 digits, about 16 bits of X).
//   cm = 1/2 sum over the index planes of the represented operands (digit sums times 2^(p-9)), cq likewise for
//   the sign plane: the -1 of the +-1 planes. um = scale log2e / lam_m, uq = scale log2e sqrt(pi/2)/d / lam_q.
__device__ __forceinline__ void tc_query_prep(const DecodeArgs& a, int b, int h, uint8_t* sm, const SFrag<kTcD>& sf) {
  constexpr int D = kTcD, NCOL = kMaxG;
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* qr = reinterpret_cast<float*>(sm + kTcPrep);
  float* qp = qr + NCOL * D;
  float* red = qp + NCOL * D;
  query_rot_proj<D, kTcThreads, 1>(a, b, h, qr, qp, red, sf);
  uint8_t* bq = sm + kTcBq;
  float* cst = reinterpret_cast<float*>(sm + kTcCst);
  if (warp < NCOL) {
    const int hd = warp;
    const bool live = hd < lv.G;
    const float wa = lv.cb[kCbW + 0], wb = lv.cb[kCbW + 1];
    float qpm = 0.f;
    for (int j = lane; j < D; j += 32) qpm = fmaxf(qpm, fabsf(qp[hd * D + j]));
    qpm = warp_max(qpm);
    const float mx = red[3 * NCOL + hd];
    const float wmax = fmaxf(fabsf(wa), fabsf(wb));
    const float lam_m = (mx > 0.f && wmax > 0.f) ? exp2f(floorf(log2f(448.f / (2.f * wmax * 512.f * mx)))) : 1.f;
    const float lam_q = qpm > 0.f ? exp2f(floorf(log2f(448.f / (2.f * 512.f * qpm)))) : 1.f;
    float sum_m = 0.f, sum_q = 0.f;
    for (int e = lane; e < 3 * D; e += 32) {  // e = (plane, coordinate)
      const int pl = e / D, j = e % D;
      int cw, kk, p;
      coord_slot(j, cw, kk, p);
      const int k = 32 * (4 * pl + cw) + kk;
      const float pre = (float)(1 << (9 - p));
      float x = 0.f;
      if (live) x = pl < 2 ? 2.f * (pl == 0 ? wa : wb) * lam_m * qr[hd * D + j] * pre : 2.f * lam_q * qp[hd * D + j] * pre;
      float rep = 0.f;
#pragma unroll
      for (int dg = 0; dg < 4; ++dg) {
        const uint8_t v = to_e4m3(x);
        const float fv = from_e4m3(v);
        x -= fv;
        rep += fv;
        bq[bq_offset(4 * hd + dg, k)] = v;
      }
      const float y = rep * (1.f / pre);  // exact: pre is a power of two
      if (pl < 2) sum_m += y;
      else sum_q += y;
    }
    sum_m = warp_sum(sum_m);
    sum_q = warp_sum(sum_q);
    if (lane == 0) {
      const float kappa = 1.2533141373155003f / (float)D;  // sqrt(pi/2) / d
      const float um = a.scale * kLog2e / lam_m, uq = a.scale * kLog2e * kappa / lam_q;
      cst[4 * hd + 0] = um;
      cst[4 * hd + 1] = um * 0.5f * sum_m;
      cst[4 * hd + 2] = uq;
      cst[4 * hd + 3] = uq * 0.5f * sum_q;
    }
  }
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // B is read by the tensor cores
  __syncthreads();
}

template <int VB, bool PAGED>
__global__ void __launch_bounds__(kTcThreads, 1) k_decode_tc(DecodeArgs a) {
  constexpr int D = kTcD, NT = kTcThreads, NB = kTcNB, STAGES = tc_stages<VB>();
  constexpr int NG = D / 32;  // value groups
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const LayerView& lv = a.lv;
  const int sp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nsp = a.plan.n_splits;
  float* part = reinterpret_cast<float*>(a.ws + a.plan.part_off +
                                         (((size_t)b * lv.Hkv + h) * (nsp + 1) + sp) * a.plan.part_stride);
  float* scratch = reinterpret_cast<float*>(sm + kTcStage);
  const int slot = row_slot(a, b);
  if (slot < 0 || slot >= lv.max_seqs) {
    pdl_wait();
    pdl_launch();
    write_empty_partial(part, D, tid, NT, kMaxG);
    finish_unit<D, NT, 1>(a, b, h, scratch);
    return;
  }
  if (sp == nsp) {
    pdl_wait();
    pdl_launch();
    const bool smem_ok = ring_split<D, NT, 1>(a, b, h, slot, part, sm);
    finish_unit<D, NT, 1>(a, b, h, scratch, smem_ok);
    return;
  }
  int L, Np, P;
  seq_packed(lv, slot, L, Np, P);
  const int n_pages = (P + kPage - 1) / kPage;
  const int pps = a.plan.pages_per_split;
  if (sp == 0 && tid == 0 && n_pages > nsp * pps) set_status(lv.status, TQ_DEV_ERR_SPLITS);
  const int pg0 = sp * pps, pg1 = min(n_pages, pg0 + pps);
  if (pg0 >= pg1) {
    pdl_wait();
    pdl_launch();
    write_empty_partial(part, D, tid, NT, kMaxG);
    finish_unit<D, NT, 1>(a, b, h, scratch);
    return;
  }
  const int npg = pg1 - pg0;
  const PageLayout pl = page_layout(D, VB, 3);
  const uint32_t PB = pl.bytes;
  TcBars* bars = reinterpret_cast<TcBars*>(sm);
  volatile int* abort_flag = &bars->abort;
  uint8_t* stage0 = sm + kTcStage;
  const uint8_t* gpages = lv.pages + ((size_t)slot * lv.Hkv + h) * lv.max_pages * PB;
  auto page_src = [&](int p) -> const uint8_t* {  // page p of this split (a missing block reads block 0)
    if (!PAGED) return gpages + (size_t)(pg0 + p) * PB;
    const int blk = lv.btab[(size_t)slot * lv.max_pages + pg0 + p];
    if ((unsigned)blk >= (unsigned)lv.n_blocks) {
      set_status(lv.status, TQ_DEV_ERR_BLOCK);
      return lv.pages + (size_t)h * PB;
    }
    return lv.pages + ((size_t)blk * lv.Hkv + h) * PB;
  };
  // wait-timeout test hook: page fault_k of this CTA gets neither its copy nor its expected-byte count, and
  // the waits for it give up after a.fault_polls polls
  const int fault_k = (a.fault_stage >= 0 && a.fault_stage < STAGES && sp == 0 && h == 0 && b == 0) ? a.fault_stage : -1;
  auto full_limit = [&](int p) { return p == fault_k ? a.fault_polls : kWaitPolls; };
  int issued = 0;  // producer: pages whose copy was issued (the hook's page counts as issued)
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 12);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&bars->a_ready[i], 4);
      mbar_init(&bars->mma_done[i], 1);
      mbar_init(&bars->s_free[i], 4);
      for (int w = 0; w < 4; ++w) {
        mbar_init(&bars->p_ready[i][w], 1);
        mbar_init(&bars->p_free[i][w], 1);
      }
    }
    bars->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    // the first pages are requested before the stream wait (inputs of this kernel are complete then)
    for (; issued < STAGES && issued < npg; ++issued) {
      if (issued == fault_k) continue;
      mbar_expect_tx(&bars->full[issued], PB);
      bulk_g2s(stage0 + (size_t)issued * PB, page_src(issued), PB, &bars->full[issued]);
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(&bars->tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    tc_fence_before();
  }
  SFrag<D> sfrag;
  sfrag_prefetch<D>(lv, sfrag);
  tc_query_prep(a, b, h, sm, sfrag);  // ends with a block barrier; barriers initialised, B ready
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  pdl_wait();  // the partials and counters of any decode that shares ws are no longer in use
  pdl_launch();

  // phase (parity) of the n-th completion of a barrier used once per round of `period` pages
  auto par = [](int p, int period) { return (uint32_t)((p / period) & 1); };
  float* alpha_s = reinterpret_cast<float*>(sm + kTcAlpha);          // [NB][4][4]
  uint16_t* pbuf = reinterpret_cast<uint16_t*>(sm + kTcP);           // [NB][4][kTcPRow]
  const float* cst = reinterpret_cast<const float*>(sm + kTcCst);    // [4][4]
  int mma_issued = 0;  // MMA thread: pages whose score MMAs were committed

  // group partials for the merge (value warp w / softmax warp w), kept in registers until after the loop
  float O[8][4];
  float m_run[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY}, l_run[4] = {0.f, 0.f, 0.f, 0.f};

  if (warp == 0) {
    // ---- producer ----
    if (lane == 0) {
      for (; issued < npg; ++issued) {
        const int s = issued % STAGES;
        if (!tc_wait(&bars->empty[s], par(issued - STAGES, STAGES), abort_flag)) break;
        mbar_expect_tx(&bars->full[s], PB);
        bulk_g2s(stage0 + (size_t)s * PB, page_src(issued), PB, &bars->full[s]);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      const uint32_t bq = smem_u32(sm + kTcBq);
      for (int p = 0; p < npg; ++p) {
        const int bi = p % NB;
        if (!tc_wait(&bars->a_ready[bi], par(p, NB), abort_flag)) break;
        if (p >= NB && !tc_wait(&bars->s_free[bi], par(p - NB, NB), abort_flag)) break;
        tc_fence_after();
        const uint32_t abase = tmem + 128u * bi, dm = abase + 96u, dq = abase + 112u;
#pragma unroll
        for (int ks = 0; ks < kTcKSteps; ++ks) {
          const uint64_t bd = desc_sw128(bq + (ks >> 2) * 2048 + (ks & 3) * 32);
          mma_e4m3_ts(ks < 8 ? dm : dq, abase + 8u * ks, bd, (ks & 7) != 0 ? 1u : 0u);
        }
        mma_commit(&bars->mma_done[bi]);
        ++mma_issued;
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---- key expanders: thread t builds A row t ----
    const int t = tid - 128;
    const int tile = t >> 4, g = t & 7, r = (t >> 3) & 1;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    for (int p = 0; p < npg; ++p) {
      const int s = p % STAGES, bi = p % NB;
      if (!tc_wait(&bars->full[s], par(p, STAGES), abort_flag, full_limit(p))) break;
      if (p >= NB && !tc_wait(&bars->mma_done[bi], par(p - NB, NB), abort_flag)) break;
      tc_fence_after();
      const uint32_t* kw = reinterpret_cast<const uint32_t*>(stage0 + (size_t)s * PB + pl.kbits_off);
#pragma unroll
      for (int plane = 0; plane < 3; ++plane) {
        uint32_t col[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t w = kw[((tile * 3 + plane) * 32 + 4 * g + c) * 2 + r];
          const uint32_t w4 = w >> 4;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            col[8 * c + q] = w & (0x01010101u << q);
            col[8 * c + 4 + q] = w4 & (0x01010101u << q);
          }
        }
        tmem_st32(tmem + lane_base + 128u * bi + 32u * plane, col);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->a_ready[bi]);
        mbar_arrive(&bars->empty[s]);
      }
    }
  } else if (warp >= 8 && warp < 12) {
    // ---- softmax: thread t = token t of the page; warp w = tokens 32w .. 32w + 31 ----
    const int w = warp - 8, t = tid - 256;
    const uint32_t lane_base = (uint32_t)(32 * w) << 16;
    float um[4], umcm[4], uq[4], uqcq[4];
#pragma unroll
    for (int hd = 0; hd < 4; ++hd) {
      um[hd] = cst[4 * hd];
      umcm[hd] = cst[4 * hd + 1];
      uq[hd] = cst[4 * hd + 2];
      uqcq[hd] = cst[4 * hd + 3];
    }
    // value position of this token's code fields: pos (2-bit: vpos2(kap, hiT); 4-bit: vpos4(hiT))
    const int tau = t & 31, kap = tau >> 4, hiT = (tau >> 3) & 1;
    const float pre = (float)(1u << (24 - (VB == 2 ? vpos2(kap, hiT) : vpos4(hiT))));
    for (int p = 0; p < npg; ++p) {
      const int s = p % STAGES, bi = p % NB;
      if (!tc_wait(&bars->mma_done[bi], par(p, NB), abort_flag)) break;
      if (!tc_wait(&bars->full[s], par(p, STAGES), abort_flag, full_limit(p))) break;  // norms, scales
      tc_fence_after();
      uint32_t acc[32];
      tmem_ld32(tmem + lane_base + 128u * bi + 96u, acc);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[bi]);
      const uint8_t* pg = stage0 + (size_t)s * PB;
      const uint32_t nw = reinterpret_cast<const uint32_t*>(pg + pl.norms_off)[t];
      const float nv = __half2float(__ushort_as_half((uint16_t)(nw & 0xffffu)));
      const float gv = __half2float(__ushort_as_half((uint16_t)(nw >> 16)));
      const int valid = P - (pg0 + p) * kPage;  // tokens of this page inside the sequence
      float sc[4];
#pragma unroll
      for (int hd = 0; hd < 4; ++hd) {
        const float am = (__uint_as_float(acc[4 * hd]) + __uint_as_float(acc[4 * hd + 1])) +
                         (__uint_as_float(acc[4 * hd + 2]) + __uint_as_float(acc[4 * hd + 3]));
        const float aq = (__uint_as_float(acc[16 + 4 * hd]) + __uint_as_float(acc[16 + 4 * hd + 1])) +
                         (__uint_as_float(acc[16 + 4 * hd + 2]) + __uint_as_float(acc[16 + 4 * hd + 3]));
        sc[hd] = t < valid ? nv * fmaf(gv, fmaf(uq[hd], aq, -uqcq[hd]), fmaf(um[hd], am, -umcm[hd])) : -INFINITY;
      }
      // largest value scale of this warp's 32 tokens (finite non-negative f16: bits order like values)
      const uint32_t* vsc = reinterpret_cast<const uint32_t*>(pg + pl.vscale_off);
      uint32_t smax_bits = 0;
      for (int i = lane; i < 16 * NG; i += 32) smax_bits = __vmaxu2(smax_bits, vsc[16 * w * NG + i]);
      smax_bits = __reduce_max_sync(0xffffffffu, max(smax_bits & 0xffffu, smax_bits >> 16));
      // p * 2^(24 - pos) <= 2^(15 - max(e2, 0)) keeps P' and P' s below 2^15 (f16)
      const float E = (float)(9 + max((int)((smax_bits >> 10) & 31u) - 14, 0));
      float pv[4], al[4];
#pragma unroll
      for (int hd = 0; hd < 4; ++hd) {
        const float mx = warp_max(sc[hd]);
        const float m_new = fmaxf(m_run[hd], mx + E);
        al[hd] = (m_new == -INFINITY) ? 1.f : exp2f(m_run[hd] - m_new);
        m_run[hd] = m_new;
        const float pn = exp2f(sc[hd] - (m_new == -INFINITY ? 0.f : m_new));  // exp2(-inf) = 0
        l_run[hd] = fmaf(l_run[hd], al[hd], pn);
        pv[hd] = pn * pre;
      }
      if (p >= NB && !tc_wait(&bars->p_free[bi][w], par(p - NB, NB), abort_flag)) break;
      uint16_t* pb = pbuf + (size_t)bi * 4 * kTcPRow;
#pragma unroll
      for (int hd = 0; hd < 4; ++hd) pb[hd * kTcPRow + t] = __half_as_ushort(__float2half_rn(pv[hd]));
      if (lane == 0) {
#pragma unroll
        for (int hd = 0; hd < 4; ++hd) alpha_s[(bi * 4 + w) * 4 + hd] = al[hd];
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->p_ready[bi][w]);
        mbar_arrive(&bars->empty[s]);
      }
    }
#pragma unroll
    for (int hd = 0; hd < 4; ++hd) l_run[hd] = warp_sum(l_run[hd]);
  } else if (warp >= 12) {
    // ---- value warps: P.V of tokens 32w .. 32w + 31, as the f16 mma.sync path of tq_decode.cu ----
    const int w = warp - 12, g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) O[mt][0] = O[mt][1] = O[mt][2] = O[mt][3] = 0.f;
    constexpr uint32_t kVmax = (1u << VB) - 1u;
    constexpr uint32_t kOff00 = voff_pattern(kVmax, VB == 2 ? vpos2(0, 0) : vpos4(0));
    constexpr uint32_t kOff01 = voff_pattern(kVmax, VB == 2 ? vpos2(0, 1) : vpos4(1));
    constexpr uint32_t kOff10 = voff_pattern(kVmax, VB == 2 ? vpos2(1, 0) : vpos4(0));
    constexpr uint32_t kOff11 = voff_pattern(kVmax, VB == 2 ? vpos2(1, 1) : vpos4(1));
    for (int p = 0; p < npg; ++p) {
      const int s = p % STAGES, bi = p % NB;
      if (!tc_wait(&bars->p_ready[bi][w], par(p, NB), abort_flag)) break;
      if (!tc_wait(&bars->full[s], par(p, STAGES), abort_flag, full_limit(p))) break;
      const uint8_t* pg = stage0 + (size_t)s * PB;
      const uint32_t* vsc = reinterpret_cast<const uint32_t*>(pg + pl.vscale_off);  // [token pair][group] f16x2
      const uint32_t* vw = reinterpret_cast<const uint32_t*>(pg + pl.vbits_off);
      const uint32_t* pb = reinterpret_cast<const uint32_t*>(pbuf + (size_t)bi * 4 * kTcPRow);
      // B fragments of P' (no value scale yet): [k-step kap][tokens 0-7 / 8-15], column g = head g
      uint32_t pbf[2][2];
#pragma unroll
      for (int kp = 0; kp < 2; ++kp)
#pragma unroll
        for (int hi = 0; hi < 2; ++hi)
          pbf[kp][hi] = g < 4 ? pb[g * (kTcPRow / 2) + 16 * w + 8 * kp + 4 * hi + c] : 0u;
      const float* al = alpha_s + (bi * 4 + w) * 4;
      const float a0 = c < 2 ? al[2 * c] : 1.f, a1 = c < 2 ? al[2 * c + 1] : 1.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_free[bi][w]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t bf[2][2];
#pragma unroll
        for (int kp = 0; kp < 2; ++kp) {
          const int tile = 2 * w + kp;
          bf[kp][0] = hmul2_u32(pbf[kp][0], vsc[(8 * tile + c) * NG + q]);
          bf[kp][1] = hmul2_u32(pbf[kp][1], vsc[(8 * tile + 4 + c) * NG + q]);
        }
        float coff[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16(coff, kOff00, kOff00, kOff01, kOff01, bf[0][0], bf[0][1]);
        mma_f16(coff, kOff10, kOff10, kOff11, kOff11, bf[1][0], bf[1][1]);
#pragma unroll
        for (int i = 0; i < 4; ++i) coff[i] *= 0.5f;
#pragma unroll
        for (int mh = 0; mh < 2; ++mh) {
          const int mt = 2 * q + mh;
          float acc[4] = {coff[0], coff[1], coff[2], coff[3]};
          if (VB == 2) {
            const uint32_t wv = vw[(w * (D / 16) + mt) * 32 + lane];
            const uint32_t w2 = wv >> 2, w6 = wv >> 6;
            mma_f16(acc, wv & 0x00030003u, w2 & 0x00030003u, wv & 0x00300030u, w6 & 0x00300030u, bf[0][0], bf[0][1]);
            mma_f16(acc, wv & 0x00C000C0u, w6 & 0x00C000C0u, wv & 0x03000300u, w6 & 0x03000300u, bf[1][0], bf[1][1]);
          } else {
            const uint2 ww = reinterpret_cast<const uint2*>(vw)[(w * (D / 16) + mt) * 32 + lane];
            const uint32_t x0 = ww.x, x8 = ww.x >> 8, y0 = ww.y, y8 = ww.y >> 8;
            mma_f16(acc, x0 & 0x000F000Fu, x8 & 0x000F000Fu, x0 & 0x00F000F0u, x8 & 0x00F000F0u, bf[0][0], bf[0][1]);
            mma_f16(acc, y0 & 0x000F000Fu, y8 & 0x000F000Fu, y0 & 0x00F000F0u, y8 & 0x00F000F0u, bf[1][0], bf[1][1]);
          }
          O[mt][0] = fmaf(O[mt][0], a0, acc[0]);
          O[mt][1] = fmaf(O[mt][1], a1, acc[1]);
          O[mt][2] = fmaf(O[mt][2], a0, acc[2]);
          O[mt][3] = fmaf(O[mt][3], a1, acc[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty[s]);
    }
  }
  // ---- after the loops: drain, free TMEM, merge the four group partials ----
  tc_fence_before();
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  bool drained = true;
  if (aborted) {
    // every copy or MMA batch that was issued is waited for (bounded) before shared memory or TMEM is
    // reused: the latest one of each stage / buffer (earlier ones were consumed before it was issued)
    if (tid == 0)
      for (int s = 0; s < STAGES; ++s) {
        const int last = s + STAGES * ((issued - 1 - s) / STAGES);  // latest page issued into stage s
        if (s < issued && last != fault_k) drained = mbar_wait(&bars->full[s], par(last, STAGES)) && drained;
      }
    if (tid == 32)
      for (int i = 0; i < NB; ++i) {
        const int last = i + NB * ((mma_issued - 1 - i) / NB);
        if (i < mma_issued) drained = mbar_wait(&bars->mma_done[i], par(last, NB)) && drained;
      }
    if (tid == 0) set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
  }
  drained = __syncthreads_and(drained) != 0;
  tc_fence_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem) : "memory");
  if (aborted) {
    write_empty_partial(part, D, tid, NT, kMaxG);
    finish_unit<D, NT, 1>(a, b, h, scratch, drained);
    return;
  }
  // group partials -> shared memory (the stages are free now)
  float* wm = scratch;           // [4 groups][4 heads]
  float* wl = wm + 16;           // [4][4]
  float* wf = wl + 16;           // [4][4] group weights
  float* wo = wf + 16;           // [4][4][D]
  if (warp >= 8 && warp < 12 && lane == 0) {
#pragma unroll
    for (int hd = 0; hd < 4; ++hd) {
      wm[(warp - 8) * 4 + hd] = m_run[hd];
      wl[(warp - 8) * 4 + hd] = l_run[hd];
    }
  }
  if (warp >= 12) {
    const int w = warp - 12, g = lane >> 2, c = lane & 3;
    if (c < 2) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int j0 = 16 * mt + g;
        wo[(w * 4 + 2 * c) * D + j0] = O[mt][0];
        wo[(w * 4 + 2 * c + 1) * D + j0] = O[mt][1];
        wo[(w * 4 + 2 * c) * D + j0 + 8] = O[mt][2];
        wo[(w * 4 + 2 * c + 1) * D + j0 + 8] = O[mt][3];
      }
    }
  }
  __syncthreads();
  if (tid < 16) {
    const int hd = tid % 4, w = tid / 4;
    float m = -INFINITY;
#pragma unroll
    for (int v = 0; v < 4; ++v) m = fmaxf(m, wm[v * 4 + hd]);
    const float mw = wm[w * 4 + hd];
    wf[w * 4 + hd] = (m == -INFINITY || mw == -INFINITY) ? 0.f : exp2f(mw - m);
  }
  __syncthreads();
  for (int i = tid; i < 4 * D; i += NT) {
    const int hd = i / D, j = i % D;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) o = fmaf(wf[w * 4 + hd], wo[(w * 4 + hd) * D + j], o);
    part[2 * 4 + hd * D + j] = o;
    if (j == 0) {
      float m = -INFINITY, l = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        m = fmaxf(m, wm[w * 4 + hd]);
        l = fmaf(wf[w * 4 + hd], wl[w * 4 + hd], l);
      }
      part[hd] = m;
      part[4 + hd] = l;
    }
  }
  __syncthreads();  // the merge scratch has been read; combine_unit reuses it
  finish_unit<D, NT, 1>(a, b, h, scratch + 16 * 3 + 4 * 4 * D);
}

template <int VB, bool PAGED>
bool tc_attr() {
  static int done = 0;  // set once, outside any stream capture that follows
  if (!done) {
    if (cudaFuncSetAttribute(k_decode_tc<VB, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc_smem_bytes<VB>()) != cudaSuccess)
      return false;
    done = 1;
  }
  return true;
}

}  // namespace

int decode_tc_setup(int vb, bool paged) {
  const bool ok = vb == 2 ? (paged ? tc_attr<2, true>() : tc_attr<2, false>())
                          : (paged ? tc_attr<4, true>() : tc_attr<4, false>());
  return ok ? 1 : -1;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, int batch, int phase, cudaStream_t s) {
  const int vb = a.lv.vb;
  const bool paged = a.lv.btab != nullptr;
  if (a.lv.d != kTcD || a.lv.kb != 3 || a.qpr != 1 || (vb != 2 && vb != 4)) return cudaErrorNotSupported;
  if (decode_tc_setup(vb, paged) < 0) return cudaErrorInvalidValue;
  if (phase == 0) {  // zero the arrival counters (every decode call leaves them at zero)
    cudaError_t e = cudaMemsetAsync(a.ws + a.plan.cnt_off, 0, sizeof(int32_t) * (size_t)batch * a.lv.Hkv, s);
    if (e != cudaSuccess) return e;
  }
  if (phase < 0 || phase == 1) {
    const dim3 grid(a.plan.n_splits + 1, a.lv.Hkv, batch);
    const size_t smem = vb == 2 ? tc_smem_bytes<2>() : tc_smem_bytes<4>();
    cudaError_t e = vb == 2 ? (paged ? launch_pdl(k_decode_tc<2, true>, grid, dim3(kTcThreads), smem, s, a)
                                     : launch_pdl(k_decode_tc<2, false>, grid, dim3(kTcThreads), smem, s, a))
                            : (paged ? launch_pdl(k_decode_tc<4, true>, grid, dim3(kTcThreads), smem, s, a)
                                     : launch_pdl(k_decode_tc<4, false>, grid, dim3(kTcThreads), smem, s, a));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace tq
