// Prefill attention over the packed history on tcgen05 tensor cores (TurboQuant vLLM guide §七, first
// item: prefill that reads the quantised cache; §三 hybrid estimator, §二 codes). A prefill chunk gives
// every KV head n_q x G query rows against the same packed pages, so here the key operands are
// expanded once per page and shared by a tile of 128 query rows (32 queries x the 4 query heads of one
// KV head), instead of by the 8 query columns of the decode kernel's mma.sync path.
//
// One CTA = one tile, one KV head, one split of the tile's visible pages. It writes one partial per
// (query, KV head, split) in the decode workspace's layout (m, l, o in the rotated basis, log2 units);
// a ring-only launch of the decode kernel then adds the exact ring tokens and combines.
//
// Scores, with the odd-symmetric 2-bit codebook c[idx] = a_h (2 h - 1) + a_l (2 l - 1) and the QJL
// sign s = 2 sigma - 1, are one fp32 accumulator in TMEM:
//   S[r][t] = A_hi . B_h + A_lo . B_h + A_hi . B_l + A_qp . B_s
//     A_hi + A_lo = lambda a_h q_rot (f16 hi + remainder), A_qp = lambda kappa (S q_rot) (f16),
//     B_h = +-1, B_l = +-rho (rho = a_l / a_h in f16), B_s = +-gamma_t (gamma_t is stored as f16),
// so S = lambda (<q_rot, c[idx_t]> + kappa gamma_t <S q_rot, s_t>) up to the f16 rounding of the l and
// QJL operands (as in the decode kernel), and the logit is S n_t scale / lambda. lambda, a power of two
// per tile, keeps the operands inside the f16 range. P (f16) and the dequantised values V^T =
// s_g (code - offset) (f16) feed the P.V MMA into a second TMEM accumulator; the softmax rescales it
// lazily (only when a row maximum grows by more than 2^8).
#include <cmath>

#include <cuda_runtime.h>

#include "tq_tcgen05.cuh"

namespace tq {
namespace {

constexpr int kPtThreads = 256;  // 8 warps: warp w covers TMEM lanes 32 (w % 4).. and column half w / 4
constexpr float kPtLog2e = 1.4426950408889634f;
// shared memory (offsets from a 1024-byte aligned base): three A tiles, three B tiles, two page stages
constexpr uint32_t kPtAhi = 0, kPtAlo = 32768, kPtAqp = 65536;
constexpr uint32_t kPtB0 = 98304, kPtB1 = 131072, kPtB2 = 163840, kPtStg = 196608;
// after the stages: per-token logit factors [128], row exchange [2][128], block maximum [8], barriers [8]
constexpr uint32_t kPtTail = 128 * 4 + 256 * 4 + 8 * 4 + 8 * 8;

struct PrefillTcArgs {
  LayerView lv;
  const uint16_t* q;       // bf16 [batch][qpr][Hq][128]
  const int32_t* seq_ids;  // [batch]
  const int32_t* n_q;      // [batch]: the row's last n_q tokens are its queries
  int qpr;                 // query slots per batch row
  float scale;             // softmax scale
  uint8_t* ws;
  DecodePlan plan;         // partial layout; n_splits history splits + the ring partial
};

__host__ __device__ constexpr size_t prefill_tc_smem(uint32_t page_bytes) {
  return 1024 + kPtStg + 2 * ((page_bytes + 127) / 128 * 128) + kPtTail;
}

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

// One bounded mbarrier wait that every thread of the CTA agrees on.
__device__ __forceinline__ bool pt_wait_all(uint64_t* bar, uint32_t parity) {
  return __syncthreads_and(mbar_wait(bar, parity)) != 0;
}

// Pairs of f16 (512 + code) from a value word: the code field at bit `pos` (and pos + 16) moved to
// mantissa bits 1.. of an f16 whose exponent puts 0.5 in the last mantissa bit.
template <int VB>
__device__ __forceinline__ uint32_t code_pair_512(uint32_t w, int pos) {
  constexpr uint32_t mask = VB == 2 ? 0x00030003u : 0x000F000Fu;
  return (((w >> pos) & mask) << 1) | 0x60006000u;
}

template <int VB>
__global__ void __launch_bounds__(kPtThreads, 1) k_prefill_tc(PrefillTcArgs a) {
  constexpr int D = 128, KB = 3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, h = blockIdx.y;
  const int S = a.plan.n_splits;
  const int b = blockIdx.z / S, split = blockIdx.z % S;
  const PageLayout pl = page_layout(D, VB, KB);
  const uint32_t PB = pl.bytes, PBS = (pl.bytes + 127) / 128 * 128;
  uint8_t* stg = sm + kPtStg;
  float* ns = reinterpret_cast<float*>(stg + 2 * PBS);  // [128] logit factor n_t scale log2e / lambda
  float* xrow = ns + 128;                                 // [2][128] row maxima / sums of the two halves
  float* bmax = xrow + 256;                               // [8] per-warp operand maxima
  uint64_t* bars = reinterpret_cast<uint64_t*>(bmax + 8);  // 0 S table, 1 projection, 2-3 pages, 4 S, 5 O
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 6);
  // this thread's query row (TMEM lane) and column half
  const int r = 32 * (warp & 3) + lane, ch = warp >> 2;
  const int qi = r >> 2, g = r & 3, qidx = 32 * tile + qi;
  pdl_wait();  // sequence state, pages and queries come from earlier work on the stream
  pdl_launch();
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
  const int npg_tile = i_last >= 32 * tile ? (vis(i_last) + kPage - 1) / kPage : 0;
  const int pps = (npg_tile + S - 1) / S;
  const int pg0 = min(npg_tile, split * pps), pg1 = min(npg_tile, pg0 + pps), n = pg1 - pg0;
  const int vis_r = vis(qidx);
  const bool row_out = qidx < a.qpr;  // a virtual row of the launch (padding rows get an empty partial)
  float* part = row_out ? reinterpret_cast<float*>(a.ws + a.plan.part_off +
                                                   ((((size_t)b * a.qpr + qidx) * lv.Hkv + h) * (S + 1) + split) *
                                                       a.plan.part_stride)
                        : nullptr;
  if (n == 0) {  // nothing visible in this split: empty partials (m = -inf, l = 0, o = 0)
    if (row_out) {
      for (int j = 64 * ch; j < 64 * ch + 64; ++j) part[2 * kMaxG + g * D + j] = 0.f;
      if (ch == 0) {
        part[g] = -INFINITY;
        part[kMaxG + g] = 0.f;
      }
    }
    return;
  }

  // ---- setup: barriers, TMEM (256 columns: S at 0, O at 128), the S table for the projection ----
  if (tid == 0) {
    for (int i = 0; i < 6; ++i) mbar_init(&bars[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    mbar_expect_tx(&bars[0], 2u * D * D);
    bulk_g2s(sm + kPtB2, lv.S_sw, 2u * D * D, &bars[0]);
    mbar_expect_tx(&bars[2], PB);  // the first page
    bulk_g2s(stg, pt_page(lv, slot, h, pg0), PB, &bars[2]);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;\n" ::"r"(smem_u32(tslot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  // ---- query rows: q_rot = Pi q (warp-per-row FWHT), bf16 hi / lo for the projection, fp32 copy ----
  float* qr = reinterpret_cast<float*>(sm + kPtB0);  // [128][128] fp32 q_rot (B0 and B1 until the pages)
  const float rs = rsqrtf((float)D);
  float amax = 0.f;
  for (int rr = warp; rr < 128; rr += 8) {
    const int i = 32 * tile + (rr >> 2), gg = rr & 3;
    float x[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = 4 * lane + e;
      x[e] = (i < nq && i < a.qpr && slot_ok)
                 ? bf16_to_f32(a.q[(((size_t)b * a.qpr + i) * lv.Hq + h * kMaxG + gg) * D + j]) * lv.D[j]
                 : 0.f;
    }
    warp_fwht<4>(x, lane);
    uint32_t hb[2], lb[2];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[e] *= rs;
      qr[rr * D + 4 * lane + e] = x[e];
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
    *reinterpret_cast<uint2*>(sm + kPtAhi + sw128_offset(rr, 4 * lane)) = make_uint2(hb[0], hb[1]);
    *reinterpret_cast<uint2*>(sm + kPtAlo + sw128_offset(rr, 4 * lane)) = make_uint2(lb[0], lb[1]);
  }
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot, t_s = tmem, t_o = tmem + 128;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  // phases armed on each barrier (a copy or an MMA batch that completes it) and seen complete, kept
  // alike by every thread, for the drain after a wait that gave up
  uint32_t armed[6] = {1, 0, 1, 0, 0, 0}, seen[6] = {0, 0, 0, 0, 0, 0};
  bool ok = pt_wait_all(&bars[0], 0);  // S table landed
  if (ok) ++seen[0];
  if (ok) ++armed[1];
  if (ok && tid == 0) {  // projection q_proj = S q_rot into TMEM columns [0, 128): A = q_rot hi, lo (bf16)
    tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      const uint32_t koff = ((ks & 7) >> 2) * 16384 + (ks & 3) * 32;
      umma_bf16(t_s, umma_desc_sw128(smem_u32(sm + (ks < 8 ? kPtAhi : kPtAlo)) + koff),
                umma_desc_sw128(smem_u32(sm + kPtB2) + koff), kIdescBf16M128N128, ks > 0);
    }
    umma_commit(&bars[1]);
  }
  ok = ok && pt_wait_all(&bars[1], 0);
  if (ok) ++seen[1];
  tc_fence_after();
  // operand scale lambda: the largest of |a_h q_rot| and |kappa q_proj| maps to [2^12, 2^13)
  const float a_h = lv.cb[kCbW + 0], a_l = lv.cb[kCbW + 1];
  const float kappa = 1.2533141373155003f / (float)D;  // sqrt(pi/2) / d
  uint32_t qpv[2][32];
#pragma unroll
  for (int i = 0; i < 32; ++i) qpv[0][i] = qpv[1][i] = 0u;
  if (ok) {
    tmem_ld32(t_s + lane_base + 64 * ch, qpv[0]);
    tmem_ld32(t_s + lane_base + 64 * ch + 32, qpv[1]);
  }
  float pmax = 0.f;
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int i = 0; i < 32; ++i) pmax = fmaxf(pmax, fabsf(__uint_as_float(qpv[u][i])));
  const float wmax = warp_max(fmaxf(fabsf(a_h) * amax, kappa * pmax));
  if (lane == 0) bmax[warp] = wmax;
  __syncthreads();
  float tmax = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tmax = fmaxf(tmax, bmax[w]);
  const float lam = tmax > 0.f ? exp2f(floorf(log2f(4096.f / tmax))) : 1.f;
  // A_qp = lambda kappa q_proj (f16); A_hi / A_lo = f16 hi / remainder of lambda a_h q_rot
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    uint32_t u4[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = 8 * m + 2 * c;
      const __half2 hv = __floats2half2_rn(lam * kappa * __uint_as_float(qpv[j >> 5][j & 31]),
                                           lam * kappa * __uint_as_float(qpv[(j + 1) >> 5][(j + 1) & 31]));
      u4[c] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    *reinterpret_cast<uint4*>(sm + kPtAqp + sw128_offset(r, 64 * ch + 8 * m)) = make_uint4(u4[0], u4[1], u4[2], u4[3]);
  }
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    uint32_t hi4[4], lo4[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = 64 * ch + 8 * m + 2 * c;
      const float x0 = lam * a_h * qr[r * D + j], x1 = lam * a_h * qr[r * D + j + 1];
      const __half2 hi = __floats2half2_rn(x0, x1);
      const float2 hf = __half22float2(hi);
      const __half2 lo = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
      hi4[c] = *reinterpret_cast<const uint32_t*>(&hi);
      lo4[c] = *reinterpret_cast<const uint32_t*>(&lo);
    }
    *reinterpret_cast<uint4*>(sm + kPtAhi + sw128_offset(r, 64 * ch + 8 * m)) = make_uint4(hi4[0], hi4[1], hi4[2], hi4[3]);
    *reinterpret_cast<uint4*>(sm + kPtAlo + sw128_offset(r, 64 * ch + 8 * m)) = make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
  }
  // constants of the B planes: +-1, +-rho (f16), and the per-token +-gamma (below)
  const __half rho_h = __float2half_rn(a_l / a_h);
  const uint32_t c_h = 0x3C003C00u, c_l = (uint32_t)__half_as_ushort(rho_h) * 0x00010001u;
  const float logit = a.scale * kPtLog2e / lam;
  constexpr float kVoff = VB == 2 ? 513.5f : 519.5f;  // 512 + the mid-rise offset 2^(VB-1) - 1/2
  const __half2 voff2 = __floats2half2_rn(kVoff, kVoff);
  float m_used = -INFINITY, l_loc = 0.f;
  for (int k = 0; k < n && ok; ++k) {
    const int pg = pg0 + k, buf = k & 1;
    uint8_t* page = stg + buf * PBS;
    if (k + 1 < n) {  // next page into the other stage (its last reader finished at the barrier below)
      if (tid == 0) {
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        mbar_expect_tx(&bars[2 + (buf ^ 1)], PB);
        bulk_g2s(stg + (buf ^ 1) * PBS, pt_page(lv, slot, h, pg + 1), PB, &bars[2 + (buf ^ 1)]);
      }
      ++armed[2 + (buf ^ 1)];
    }
    ok = pt_wait_all(&bars[2 + buf], (k >> 1) & 1);
    if (ok) ++seen[2 + buf];
    if (ok && k > 0) {  // the previous P.V MMAs have read B0 and B1
      ok = pt_wait_all(&bars[5], (k - 1) & 1);
      if (ok) ++seen[5];
    }
    if (!ok) break;
    tc_fence_after();
    // ---- key planes: token tk, coordinate chunks 8 hv .. 8 hv + 7 ----
    {
      const int tk = tid >> 1, hv = tid & 1;
      const uint32_t* kw = reinterpret_cast<const uint32_t*>(page + pl.kbits_off);
      const uint32_t nw = reinterpret_cast<const uint32_t*>(page + pl.norms_off)[tk];
      const uint32_t c_s = (nw >> 16) * 0x00010001u;  // gamma_t in both halves
      if (hv == 0) ns[tk] = __half2float(__ushort_as_half((uint16_t)(nw & 0xffffu))) * logit;
      const int tl = tk >> 4, g8 = tk & 7, rr = (tk >> 3) & 1;
#pragma unroll
      for (int p = 0; p < KB; ++p) {
        uint32_t w[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) w[c] = kw[((tl * KB + p) * 32 + 4 * g8 + c) * 2 + rr];
        const uint32_t cst = p == 0 ? c_h : p == 1 ? c_l : c_s;
        uint8_t* base = sm + (p == 0 ? kPtB0 : p == 1 ? kPtB1 : kPtB2);
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) {
          const int m = 8 * hv + mm;
          uint32_t u4[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) u4[c] = (~(w[c] << (15 - m)) & 0x80008000u) | cst;  // bit 1 -> +, 0 -> -
          *reinterpret_cast<uint4*>(base + sw128_offset(tk, 8 * m)) = make_uint4(u4[0], u4[1], u4[2], u4[3]);
        }
      }
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // S = A_hi B_h + A_lo B_h + A_hi B_l + A_qp B_s
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 32; ++ks) {
        const int blkk = ks >> 3, kk = ks & 7;
        const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t aoff = blkk == 0 || blkk == 2 ? kPtAhi : blkk == 1 ? kPtAlo : kPtAqp;
        const uint32_t boff = blkk <= 1 ? kPtB0 : blkk == 2 ? kPtB1 : kPtB2;
        umma_bf16(t_s, umma_desc_sw128(smem_u32(sm + aoff) + koff), umma_desc_sw128(smem_u32(sm + boff) + koff),
                  kIdescF16M128N128, ks > 0);
      }
      umma_commit(&bars[4]);
    }
    ++armed[4];
    ok = pt_wait_all(&bars[4], k & 1);
    if (!ok) break;
    ++seen[4];
    tc_fence_after();
    // ---- softmax of row r over tokens 64 ch .. 64 ch + 63 ----
    uint32_t sv[2][32];
    tmem_ld32(t_s + lane_base + 64 * ch, sv[0]);
    tmem_ld32(t_s + lane_base + 64 * ch + 32, sv[1]);
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = 64 * ch + 32 * u + i;
        const float s = pg * kPage + t < vis_r ? __uint_as_float(sv[u][i]) * ns[t] : -INFINITY;
        sv[u][i] = __float_as_uint(s);
        mx = fmaxf(mx, s);
      }
    xrow[128 * ch + r] = mx;
    __syncthreads();
    mx = fmaxf(mx, xrow[128 * (ch ^ 1) + r]);
    // the row maximum grew by more than 2^8: move to the new maximum (O and l scaled by alpha). The TMEM
    // loads and stores are warp-wide, so a warp rescales when any of its rows needs it (alpha = 1 for the rest)
    const bool grow = mx > m_used + 8.f;
    const float alpha = !grow ? 1.f : (m_used == -INFINITY ? 0.f : exp2f(m_used - mx));
    if (__any_sync(0xffffffffu, grow && k > 0)) {
      uint32_t ov[32];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        tmem_ld32(t_o + lane_base + 64 * ch + 32 * u, ov);
#pragma unroll
        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
        tmem_st32(t_o + lane_base + 64 * ch + 32 * u, ov);
      }
    }
    if (grow) {
      l_loc *= alpha;
      m_used = mx;
    }
#pragma unroll
    for (int mm = 0; mm < 8; ++mm) {
      uint32_t u4[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = 8 * mm + 2 * c;
        const float s0 = __uint_as_float(sv[i >> 5][i & 31]), s1 = __uint_as_float(sv[(i + 1) >> 5][(i + 1) & 31]);
        const float p0 = m_used == -INFINITY ? 0.f : exp2f(s0 - m_used);
        const float p1 = m_used == -INFINITY ? 0.f : exp2f(s1 - m_used);
        l_loc += p0 + p1;
        const __half2 ph = __floats2half2_rn(p0, p1);
        u4[c] = *reinterpret_cast<const uint32_t*>(&ph);
      }
      *reinterpret_cast<uint4*>(sm + kPtB0 + sw128_offset(r, 64 * ch + 8 * mm)) = make_uint4(u4[0], u4[1], u4[2], u4[3]);
    }
    // ---- values: V^T[coordinate j][token] = s_g (code - offset), tokens 64 th .. 64 th + 63 ----
    {
      const int j = tid >> 1, th = tid & 1;
      const int mt = j >> 4, g8 = j & 7, rowhi = (j >> 3) & 1, grp = j >> 5;
      const uint32_t* vw = reinterpret_cast<const uint32_t*>(page + pl.vbits_off);
      const uint32_t* vsc = reinterpret_cast<const uint32_t*>(page + pl.vscale_off);  // [token pair][group] f16x2
#pragma unroll
      for (int mm = 0; mm < 8; ++mm) {
        const int m = 8 * th + mm, blk = m >> 2, kap = (m >> 1) & 1, hiT = m & 1, rr = rowhi + 2 * hiT;
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
        *reinterpret_cast<uint4*>(sm + kPtB1 + sw128_offset(j, 8 * m)) = make_uint4(u4[0], u4[1], u4[2], u4[3]);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // O += P V: A = P [rows x tokens] (B0), B = V^T [coordinates x tokens] (B1)
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (ks >> 2) * 16384 + (ks & 3) * 32;
        umma_bf16(t_o, umma_desc_sw128(smem_u32(sm + kPtB0) + koff), umma_desc_sw128(smem_u32(sm + kPtB1) + koff),
                  kIdescF16M128N128, (k > 0 || ks > 0) ? 1u : 0u);
      }
      umma_commit(&bars[5]);
    }
    ++armed[5];
  }
  if (ok && armed[5] > seen[5]) {
    ok = pt_wait_all(&bars[5], (armed[5] - 1) & 1);
    if (ok) ++seen[5];
  }
  tc_fence_after();
  // ---- the partial of row r: m (log2 units), l, o (rotated basis, relative to m) ----
  xrow[128 * ch + r] = l_loc;
  __syncthreads();
  const float l_row = l_loc + xrow[128 * (ch ^ 1) + r];
  const bool has = ok && m_used != -INFINITY;  // this row saw a token
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    uint32_t ov[32];
    if (ok) tmem_ld32(t_o + lane_base + 64 * ch + 32 * u, ov);  // warp-wide (ok is the same in every thread)
#pragma unroll
    for (int i4 = 0; i4 < 8 && row_out; ++i4)
      *reinterpret_cast<float4*>(part + 2 * kMaxG + g * D + 64 * ch + 32 * u + 4 * i4) =
          has ? make_float4(__uint_as_float(ov[4 * i4]), __uint_as_float(ov[4 * i4 + 1]),
                            __uint_as_float(ov[4 * i4 + 2]), __uint_as_float(ov[4 * i4 + 3]))
              : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (row_out) {
    if (ch == 0) {
      part[g] = has ? m_used : -INFINITY;
      part[kMaxG + g] = has ? l_row : 0.f;
    }
  }
  if (!ok && tid == 0) {
    // a wait gave up: nothing more is issued; wait (bounded) for every armed phase not seen complete - the
    // MMA batches before TMEM is freed, the copies before the CTA leaves its shared memory
    set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
    for (int i = 0; i < 6; ++i)
      for (uint32_t ph = seen[i]; ph < armed[i]; ++ph) mbar_wait(&bars[i], ph & 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;\n" ::"r"(tmem) : "memory");
}

}  // namespace

bool prefill_tc_eligible(const tq_ctx* ctx) {
  const tq_config& c = ctx->cfg;
  return c.head_dim == 128 && c.key_bits == 3 && c.n_q_heads == kMaxG * c.n_kv_heads;
}

int prefill_tc_splits(const tq_ctx* ctx, int batch, int q_per_row, int max_ctx_hint) {
  const int hint = (max_ctx_hint <= 0 || max_ctx_hint > ctx->cfg.max_ctx) ? ctx->cfg.max_ctx : max_ctx_hint;
  const int max_pages = std::max(1, (hint + kPage - 1) / kPage);
  const int ctas = (q_per_row + 31) / 32 * ctx->cfg.n_kv_heads * batch;
  const int sms = ctx->sm_count > 0 ? ctx->sm_count : 152;
  return std::max(1, std::min(max_pages, sms / std::max(1, ctas)));
}

cudaError_t launch_prefill_tc(const tq_ctx* ctx, int layer, const void* q, const int32_t* seq_ids, const int32_t* n_q,
                              int batch, int q_per_row, float scale, void* ws, const DecodePlan& plan, cudaStream_t s) {
  PrefillTcArgs a;
  a.lv = layer_view(ctx, layer);
  a.q = static_cast<const uint16_t*>(q);
  a.seq_ids = seq_ids;
  a.n_q = n_q;
  a.qpr = q_per_row;
  a.scale = scale;
  a.ws = static_cast<uint8_t*>(ws);
  a.plan = plan;
  const dim3 grid((q_per_row + 31) / 32, a.lv.Hkv, batch * plan.n_splits);
  const size_t smem = prefill_tc_smem(a.lv.page_bytes);
  if (smem > kMaxSmemPerCta) return cudaErrorInvalidValue;
  if (a.lv.vb == 2) {
    static bool attr = false;  // set once, outside any stream capture that follows
    if (!attr) {
      cudaError_t e = cudaFuncSetAttribute(k_prefill_tc<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr = true;
    }
    return launch_pdl(k_prefill_tc<2>, grid, dim3(kPtThreads), smem, s, a);
  }
  static bool attr4 = false;
  if (!attr4) {
    cudaError_t e = cudaFuncSetAttribute(k_prefill_tc<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr4 = true;
  }
  return launch_pdl(k_prefill_tc<4>, grid, dim3(kPtThreads), smem, s, a);
}

}  // namespace tq
