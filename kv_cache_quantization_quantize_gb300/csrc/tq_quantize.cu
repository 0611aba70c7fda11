// Quantize-on-append ([Guide] §二, five-step pipeline). Two paths write packed pages (128 tokens of
// one KV head):
//   - CUDA-core kernels (four 32-token CTAs per page) for ring flushes, decode-sized appends and f32
//     inputs; their QJL projection z = S r is an f16 mma.sync GEMM per block;
//   - persistent tcgen05 kernels for bulk bf16 appends at head_dim 64 and 128 (below) and 256
//     (tq_quantize256.cu), with the rotation and the projection on the tensor cores.
#include <algorithm>
#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "tq_quantize_common.cuh"
#include "tq_tcgen05.cuh"

namespace tq {

// tq_debug_append_wait_fault: the page task whose TMA copy the tcgen05 coders skip (-1: none) and the polls
// of its wait
std::atomic<int> g_qfault_task{-1};
std::atomic<int> g_qfault_polls{0};

namespace {

// full_tq appends: codes tokens [t_lo, t_hi) of page pg (page-relative, one 32-token block at most)
// and writes only their bits. Key words, {n, gamma} and value scales belong to one token each; a value
// word holds the codes of 8 tokens of its block, so it is read, the new tokens' fields replaced, and
// written back (one thread per word: this CTA is the block's only writer). Run by all kQThreads threads.
template <int D, int KB>
__device__ __forceinline__ void quantize_new_tokens(const AppendArgs& a, int b, int h, int slot, int L, int Np,
                                                    int pg, int t_lo, int t_hi, uint8_t* smem) {
  constexpr int HALVES = D >= 128 ? D / 128 : 1;  // 128-coordinate halves (head_dim 64: see below)
  const QSmem<D> sm(smem);
  code_tokens<D, KB>(a, b, h, slot, L, Np, pg, t_hi, t_lo, t_hi, sm);
  const int tid = threadIdx.x;
  const LayerView& lv = a.lv;
  const int vb = lv.vb, ntok = t_hi - t_lo;
  const int tb = t_lo & ~31;  // the block's first token (row 0 of the shared-memory arrays)
  uint8_t* page = page_addr(lv, slot, h, pg);
  if (!page) {  // paged cache without a block for this page: nothing is written
    if (tid == 0) set_status(lv.status, TQ_DEV_ERR_BLOCK);
    return;
  }
  const PageLayout pl = page_layout(D, vb, KB);
  uint32_t* kw = reinterpret_cast<uint32_t*>(page + pl.kbits_off);
  if (D == 64) {  // a word holds two tokens (both tiles of the block): replace the new tokens' fields
    const int grp = t_lo >> 5;
    for (int w = grp * 64 * KB + tid; w < (grp + 1) * 64 * KB; w += kQThreads) {
      const int r = w & 1, ln = (w >> 1) & 31, pi = (w >> 6) % KB;
      uint32_t mask = 0, bits = 0;
#pragma unroll
      for (int kap = 0; kap < 2; ++kap) {
        const int t = 32 * grp + 16 * kap + (ln >> 2) + 8 * r;
        if (t >= t_lo && t < t_hi) {
          mask |= 0x00FF00FFu << (8 * kap);
          bits |= kbits_field(sm.kcode + (t - tb) * D + 2 * (ln & 3), pi, KB, 4, 8 * kap);
        }
      }
      if (mask) kw[w] = (kw[w] & ~mask) | bits;
    }
  }
  for (int i = tid; D >= 128 && i < ntok * 4 * KB * HALVES; i += kQThreads) {  // (token, plane, half, c)
    const int c = i & 3, hf = (i >> 2) % HALVES, pi = (i / (4 * HALVES)) % KB, t = t_lo + i / (4 * KB * HALVES);
    const int tile = t >> 4, g = t & 7, r = (t >> 3) & 1;
    kw[((((tile * KB + pi) * HALVES + hf) * 32) + 4 * g + c) * 2 + r] =
        kbits_field(sm.kcode + (t - tb) * D + 128 * hf + 2 * c, pi, KB, 8, 0);
  }
  uint32_t* nw = reinterpret_cast<uint32_t*>(page + pl.norms_off);
  for (int t = t_lo + tid; t < t_hi; t += kQThreads) nw[t] = sm.norms[t - tb];
  uint32_t* vw = reinterpret_cast<uint32_t*>(page + pl.vbits_off);
  const int blk = t_lo >> 5;
  if (vb == 2) {
    for (int w = blk * (D / 16) * 32 + tid; w < (blk + 1) * (D / 16) * 32; w += kQThreads) {
      const int ln = w & 31, mt = (w >> 5) % (D / 16);
      const int g = ln >> 2, c = ln & 3;
      uint32_t mask = 0, bits = 0;
#pragma unroll
      for (int kap = 0; kap < 2; ++kap)
#pragma unroll
        for (int rg = 0; rg < 4; ++rg)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int t = 32 * blk + 16 * kap + 8 * (rg >> 1) + 2 * c + e;
            if (t >= t_lo && t < t_hi) {
              const int sh = 16 * e + 2 * vfield2(kap, rg);
              mask |= 3u << sh;
              bits |= (uint32_t)sm.vcode[(t - tb) * D + 16 * mt + 8 * (rg & 1) + g] << sh;
            }
          }
      if (mask) vw[w] = (vw[w] & ~mask) | bits;
    }
  } else {
    for (int w = blk * (D / 16) * 64 + tid; w < (blk + 1) * (D / 16) * 64; w += kQThreads) {
      const int kap = w & 1, ln = (w >> 1) & 31, mt = (w >> 6) % (D / 16);
      const int g = ln >> 2, c = ln & 3;
      uint32_t mask = 0, bits = 0;
#pragma unroll
      for (int rg = 0; rg < 4; ++rg)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 32 * blk + 16 * kap + 8 * (rg >> 1) + 2 * c + e;
          if (t >= t_lo && t < t_hi) {
            const int sh = 16 * e + 4 * vfield4(rg);
            mask |= 15u << sh;
            bits |= (uint32_t)sm.vcode[(t - tb) * D + 16 * mt + 8 * (rg & 1) + g] << sh;
          }
        }
      if (mask) vw[w] = (vw[w] & ~mask) | bits;
    }
  }
  uint16_t* sw = reinterpret_cast<uint16_t*>(page + pl.vscale_off);
  for (int i = t_lo * (D / 32) + tid; i < t_hi * (D / 32); i += kQThreads)
    sw[vscale_idx(D, i / (D / 32), i % (D / 32))] = sm.scales[i - tb * (D / 32)];
}

template <int D, int KB>
__global__ void __launch_bounds__(kQThreads) k_quantize_pages(AppendArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int b = blockIdx.x, h = blockIdx.y;
  pdl_wait();  // sequence state, ring and inputs come from earlier work on the stream
  pdl_launch();
  int slot, L, Np, pg, valid;
  const int j = blockIdx.z >> 2;  // 4 CTAs per page, one per 32-token block
  if (!page_task(a, b, j, slot, L, Np, pg, valid, h == 0 && blockIdx.z == 0 && threadIdx.x == 0)) return;
  quantize_page_cta<D, KB>(a, b, h, slot, L, Np, pg, valid, blockIdx.z & 3, smem);
}

// Writes the ring rows of positions [p0, L2) of row b (every KV head, K and V) from the new input,
// whose first token is position L; the ring then starts at position Np2. Run by all threads of a CTA.
__device__ __forceinline__ void write_ring_rows(const AppendArgs& a, int b, int slot, int L, int Np2, int p0, int L2) {
  const LayerView& lv = a.lv;
  const int d = lv.d, q4 = d / 4;
  const int n_items = (L2 - p0) * lv.Hkv * 2 * q4;  // (pos, head, which, quad)
  for (int it = threadIdx.x; it < n_items; it += blockDim.x) {
    const int quad = it % q4;
    int rest = it / q4;
    const int which = rest & 1;
    rest >>= 1;
    const int hh = rest % lv.Hkv, pos = p0 + rest / lv.Hkv;
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
}

// Appends of fewer than 128 tokens per row in one launch. CTA (row b, KV head h, block q) codes
// 32-token block q of the 128-token block that the append completes (if any; the ring keeps those
// tokens until the next token starts a new ring block). The last of the row's 4 Hkv CTAs to arrive
// writes the new ring rows of every head (all CTAs have read the old ones by then) and publishes the
// new length; without a block to code CTA (b, 0, 0) does that alone. When a page is coded, the ring
// starts a new block, or in full_tq mode, dependents (the decode) are released only after that, so
// they may read the state before their own stream wait; otherwise they are released at once, since
// the packed count they read then is the same before and after this append.
template <int D, int KB>
__global__ void __launch_bounds__(kQThreads) k_append_small(AppendArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_last;
  const int b = blockIdx.x, h = blockIdx.y, q32 = blockIdx.z, tid = threadIdx.x;
  pdl_wait();  // sequence state, ring and inputs come from earlier work on the stream
  const LayerView& lv = a.lv;
  const int slot = a.seq_ids[b];
  const bool first = h == 0 && q32 == 0 && tid == 0;
  if (slot < 0 || slot >= lv.max_seqs) {
    if (first) set_status(lv.status, TQ_DEV_ERR_SEQ_ID);
    return;
  }
  const int L = lv.state[2 * slot], F = lv.state[2 * slot + 1];
  const int Np = L > 0 ? kPage * ((L - 1) / kPage) : 0;
  const int nn = new_count(a, b);
  const int L2 = L + nn;
  if (nn < 0 || nn > a.max_new || L2 > lv.max_ctx) {
    if (first) set_status(lv.status, TQ_DEV_ERR_CAPACITY);
    return;
  }
  const int Np2 = L2 > 0 ? kPage * ((L2 - 1) / kPage) : 0;
  const bool code = kPage * (L2 / kPage) > kPage * (L / kPage);  // the append completes a block
  const bool roll = Np2 > Np;                                      // the ring starts a new block
  if (!a.full && !code) {
    // no page to code (the common decode step): nothing reads the old ring rows, so CTA (b, 0, 0)
    // writes every head's new rows and the length on its own and the others leave at once.
    // Dependents are released first unless the ring rolls over: the packed count (what a decode split
    // reads before its own stream wait) then does not change, and a decode's ring split waits for
    // this grid to finish.
    if (!roll) pdl_launch();
    if (h == 0 && q32 == 0) {
      write_ring_rows(a, b, slot, L, Np2, L, L2);
      __syncthreads();
      if (tid == 0) {
        lv.state[2 * slot] = L2;
        if (roll) lv.state[2 * slot + 1] = 0;
        __threadfence();
      }
      __syncthreads();
    }
    if (roll) pdl_launch();
    return;
  }
  if (a.full) {
    // full_tq: the new tokens are coded into the page that holds them. A page that this append enters
    // is coded whole (its tokens past L2 as zero vectors until they arrive), so that decode never reads
    // a block that no append has written; in an older page only the new tokens' bits are written.
    const bool entered = Np2 >= L;
    const int end_blk = entered ? Np2 / 32 + 3 : (L2 - 1) / 32;
    for (int blk = L / 32 + q32; blk <= end_blk; blk += 4) {
      const int pg = blk / 4;
      if (entered && pg * kPage == Np2) {
        quantize_page_cta<D, KB>(a, b, h, slot, L, Np, pg, min(kPage, L2 - pg * kPage), blk & 3, smem);
      } else {
        const int base = pg * kPage;
        quantize_new_tokens<D, KB>(a, b, h, slot, L, Np, pg, max(L, 32 * blk) - base,
                                   min(L2, 32 * blk + 32) - base, smem);
      }
      __syncthreads();  // shared memory is staged again by the next block
    }
  } else if (code) {
    quantize_page_cta<D, KB>(a, b, h, slot, L, Np, Np / kPage, kPage, q32, smem);  // L is inside block Np / 128
  }
  __syncthreads();  // this CTA has read the old ring rows it needed
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(lv.acnt + slot, 1);
    s_last = old == 4 * lv.Hkv - 1;
  }
  __syncthreads();
  if (s_last) {
    write_ring_rows(a, b, slot, L, Np2, max(L, Np2), L2);
    __syncthreads();
    if (tid == 0) {
      lv.acnt[slot] = 0;
      lv.state[2 * slot] = L2;
      lv.state[2 * slot + 1] = a.full ? L2 - Np2 : (roll ? 0 : F);
      __threadfence();
    }
    __syncthreads();
  }
  pdl_launch();
}

// =============================================================================================
// Bulk quantise (head_dim 64 and 128) on tcgen05 tensor cores. One persistent CTA per SM walks its pages:
//   - The bf16 K and V rows of the next page stream into shared memory (cp.async, 128-byte swizzled
//     K-major tiles) while the current page is coded.
//   - Rotation: y' = (H diag(D)) x for all 128 tokens of K and of V as two M = 128, N = K = D MMAs
//     (the +-1 entries are exact in bf16, products are exact, fp32 accumulation) into TMEM.
//   - Warps 0-7 code the keys, two threads per token row, from TMEM: norm, Lloyd-Max index,
//     residual, bf16 hi + lo split of the residual (written over the consumed K tile); then thread 0
//     issues the QJL projection z = S r as 2 D / 16 more MMAs (|r - hi - lo| <= 2^-18 |r|).
//   - Warps 8-15 code the values the same way (groups of 32, fp16 scale, mid-rise codes) and then
//     take the signs of z, so the key warps need not wait for the projection.
//   - Key words, norms and value scales go to the page straight from registers; value codes are
//     staged in shared memory for the fragment-major value layout.
// =============================================================================================
// Shared memory of the head_dim-D coder (D = 64 or 128), byte offsets: H diag(D) and S (2 D^2 each), two page
// buffers [K tile | V tile] of 128 x D bf16 each, the value codes [128][D] u8, the half-row exchange, and
// the mbarriers [8] (slot 6 holds the TMEM address) with the arming and completion counts of each barrier
// ([8] + [8] u32, see bulk_drain).
template <int D> struct QbLayout {
  static constexpr uint32_t kTile = 128u * D * 2;  // one 128 x D bf16 tile
  static constexpr uint32_t kBufBytes = 2 * kTile;
  static constexpr uint32_t kHD = 0, kS = 2u * D * D, kBuf = 4u * D * D;
  static constexpr uint32_t kVcode = kBuf + 2 * kBufBytes;
  static constexpr uint32_t kX = kVcode + 128u * D;
  static constexpr uint32_t kBar = kX + 2048 + 6144 + 2048, kEnd = kBar + 128;
  static constexpr size_t kSmem = kEnd + 1024;  // + alignment slack for the 1024-byte swizzle atoms
};
static_assert(QbLayout<128>::kSmem == 224384 && QbLayout<64>::kBuf % 1024 == 0, "layouts");
// two head_dim-64 CTAs per SM: 2 x (dynamic + 1 KB reserved) within the 228 KB of an SM
static_assert(2 * (QbLayout<64>::kSmem + 1024) <= 233472, "two CTAs per SM at head_dim 64");
// Chunk swizzle of the value-code staging rows (16-byte chunk c of row t at chunk c ^ vsw(t)): conflict-free
// row writes for 128-byte rows (D = 128) and for 64-byte rows (D = 64, two rows per 128 bytes).
template <int D> __device__ __forceinline__ int vsw(int t) { return D == 128 ? (t & 7) : ((t >> 1) & 3); }

// Loads page pg's K and V rows (bf16) into buffer `buf` (K tile at 0, V tile at 128 D 2 bytes; each D / 64
// 16 KB swizzle atoms of 64 coordinates). Pages made of new input only are fetched by 2 D / 64 TMA tensor
// copies (tensor [batch][max_new][Hkv][D], box 64 x 1 x 128 x 1, 128-byte swizzle) that complete on
// `bar`; returns true then. Pages that start in the ring are copied with plain loads and stores by
// all threads (at most one page per row and append).
// The copy is made by the nthr threads whose index relative to `first` is in [0, nthr).
// `armed` counts the copies armed on `bar` (see bulk_drain). skip (test hook): a TMA copy is not issued
// at all (no expected bytes either), so its wait gives up.
template <int D>
__device__ __forceinline__ bool bulk_tc_load(const AppendArgs& a, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                             int b, int h, int slot, int L, int Np, int pg, uint8_t* buf,
                                             uint64_t* bar, uint32_t* armed, int first, int nthr, bool skip = false) {
  constexpr int NB = D / 64;  // boxes (64-coordinate atoms) per tile
  const int rel = (int)threadIdx.x - first;
  if (rel < 0 || rel >= nthr) return pg * kPage >= L;
  if (pg * kPage >= L) {
    if (rel == 0 && !skip) {
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      mbar_expect_tx(bar, 2u * NB * 16384u);
      ++*armed;
      const int z = pg * kPage - L;
#pragma unroll
      for (int i = 0; i < 2 * NB; ++i) {
        const CUtensorMap* m = i < NB ? tmk : tmv;
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(
                smem_u32(buf + i * 16384)),
            "l"(reinterpret_cast<uint64_t>(m)), "r"(64 * (i % NB)), "r"(h), "r"(z), "r"(b), "r"(smem_u32(bar))
            : "memory");
      }
    }
    return true;
  }
  for (int q = rel; q < 2 * kPage * (D / 8); q += nthr) {
    const int which = q / (kPage * (D / 8)), t = (q / (D / 8)) % kPage, c = q % (D / 8);
    const int pos = pg * kPage + t;
    const uint16_t* src;
    if (pos < L) {
      src = a.lv.ring + ((((size_t)slot * a.lv.Hkv + h) * 2 + which) * kPage + (pos - Np)) * D;
    } else {
      src = static_cast<const uint16_t*>(which ? a.v : a.k) + (((size_t)b * a.max_new + (pos - L)) * a.lv.Hkv + h) * D;
    }
    *reinterpret_cast<uint4*>(buf + which * QbLayout<D>::kTile + sw128_offset(t, 8 * c)) =
        *reinterpret_cast<const uint4*>(src + 8 * c);
  }
  return false;
}

// kind::f16 instruction descriptor, bf16 operands, f32 accumulator, M = 128, N = D.
template <int D>
constexpr uint32_t kIdescBf16M128 = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(D >> 3) << 17) | ((128u >> 4) << 24);

// Rotation of the K and V tiles of one page (buffer at smem address buf) by the tensor cores:
// D[t][i] = sum_j x[t][j] (H D)[i][j], K into TMEM columns [0, D) of `tcol`, V into [D, 2 D).
template <int D>
__device__ __forceinline__ void bulk_tc_rotate(uint32_t tcol, uint32_t buf, uint32_t hd_addr, uint64_t* bar,
                                               uint32_t* armed) {
  tc_fence_after();
  const uint32_t xa = umma_desc_sw128_lo(buf), hb = umma_desc_sw128_lo(hd_addr);
#pragma unroll
  for (int part = 0; part < 2; ++part)  // K, then V (+one tile = 16 D descriptor units)
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint32_t koff = (ks >> 2) * 1024u + (ks & 3) * 2u;  // atom 16 KB, k step 32 B, in 16-byte units
      umma_bf16_lo(tcol + (uint32_t)D * part, xa + part * (16u * D) + koff, hb + koff, kIdescBf16M128<D>, ks > 0);
    }
  umma_commit(bar);
  ++*armed;
}

// D = head_dim (64 or 128). KB = key bits: 3 (2-bit Lloyd-Max index + sign) or 4 (3-bit index + sign,
// served with 4-bit values). TPT = threads per token row and role: 2 (512 threads, each a column half; one
// CTA per SM) or 1 (256 threads, each a whole row; at head_dim 64 two CTAs share an SM).
template <int D, int KB, int TPT>
__global__ void __launch_bounds__(256 * TPT, TPT == 1 ? 2 : 1)
    k_quantize_bulk_tc(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, AppendArgs a,
                       int pages_per_row, int batch) {
  using Lq = QbLayout<D>;
  constexpr int NT = 256 * TPT;     // threads: key warps, then value warps
  constexpr int HT = 128 * TPT;     // threads of one role
  constexpr int VL = HT;            // the value warps' leader (issues their copies and rotations, counts their waits)
  constexpr int MB = KB - 1;        // index bits = index planes
  constexpr int HC = D / TPT;       // coordinates (TMEM columns) of one thread: its token row, or a column half
  constexpr int PS = D / 16;        // bit positions between the two column halves' coordinates in a key word
  constexpr uint32_t TH = 2u * D;   // TMEM columns of one page half: [rotated K (then z = S r) | rotated V]
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* vcode = sm + Lq::kVcode;
  uint64_t* bar_tab = reinterpret_cast<uint64_t*>(sm + Lq::kBar);
  // QJL projections of pages in buffers 0 / 1: two barriers, so that a projection can never complete
  // twice before the value warps wait for it
  auto bar_qjl2 = [bar_tab](uint32_t i) { return i ? bar_tab + 7 : bar_tab + 1; };
  uint64_t* bar_ld = bar_tab + 2;   // [2]: page loads into buffer 0 / 1
  uint64_t* bar_rot = bar_tab + 4;  // [2]: rotations into TMEM half 0 / 1
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_tab + 6);
  // phases armed on barrier i and seen complete by the thread that counts it: barrier 0 (tables) and the
  // rotations by thread 0; the page loads by the thread that waits for them (0 for the first, the value
  // leader after); the QJL projections by the value leader
  uint32_t* armed = reinterpret_cast<uint32_t*>(bar_tab + 8);
  uint32_t* done = armed + 8;
  auto qjl_idx = [](uint32_t i) { return i ? 7 : 1; };
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_launch();
  if (tid == 0) {
    for (int i = 0; i < 16; ++i) armed[i] = 0u;  // armed[8], done[8]
    for (int i = 0; i < 8; ++i)
      if (i != 6) mbar_init(bar_tab + i, 1);  // slot 6 holds the TMEM address
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    mbar_expect_tx(bar_tab, 4u * D * D);
    armed[0] = 1u;
    bulk_g2s(sm + Lq::kHD, lv.HD_sw, 2u * D * D, bar_tab);
    bulk_g2s(sm + Lq::kS, lv.S_sw, 2u * D * D, bar_tab);
  }
  if (warp == 0) {  // 4 D TMEM columns: two halves of [rotated K (then z = S r) | rotated V], by page parity
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tslot)),
                 "n"(4 * D)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t hd_addr = smem_u32(sm + Lq::kHD), s_addr = smem_u32(sm + Lq::kS), buf0 = smem_u32(sm + Lq::kBuf);
  const int ntasks = batch * lv.Hkv * pages_per_row;
  int b, h, slot, L, Np, pg;
  RowTask rc;  // this thread's cached row lookup
  int cur = bulk_next(a, blockIdx.x, ntasks, pages_per_row, rc, b, h, slot, L, Np, pg);
  __syncthreads();  // barriers initialised
  bool ld_skipped = cur == a.fault_task;  // the wait-timeout test hook: this page's copy is not issued
  bool tma_cur = cur < ntasks && bulk_tc_load<D>(a, &tmk, &tmv, b, h, slot, L, Np, pg, sm + Lq::kBuf, bar_ld, armed + 2,
                                                 0, NT, ld_skipped);
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  const bool tab_ok = mbar_wait(bar_tab, 0);
  if (tid == 0 && tab_ok) ++done[0];
  bool ok = __syncthreads_and(tab_ok) != 0;
  // parities of the next wait: bit i of ph_ld / ph_rot for buffer / TMEM half i
  uint32_t ph_rot = 0, ph_qjl = 0, bufi = 0, ph_ld = 0;
  // Pipeline. Page i lives in smem buffer i % 2 and TMEM half i % 2.
  //   - The key warps code page i and issue its QJL MMAs.
  //   - The value warps first take the QJL signs of page i - 1 (its MMAs ran during the end of iteration
  //     i - 1), which frees buffer and TMEM half (i + 1) % 2. They then start the copy of page i + 1,
  //     code the values of page i, and issue the rotation of page i + 1.
  // So no warp waits on the tensor cores inside an iteration: the rotation of page i + 1 and the
  // projection of page i run while the values of page i are packed. The first page's rotation is
  // issued here.
  if (ok && cur < ntasks && tid == 0) {
    if (tma_cur) {
      if (mbar_wait(bar_ld, 0, ld_skipped ? a.fault_polls : kWaitPolls)) ++done[2];
      else ok = false;
    }
    if (ok) bulk_tc_rotate<D>(tmem, smem_u32(sm + Lq::kBuf), smem_u32(sm + Lq::kHD), bar_rot, armed + 4);
  }
  if (tma_cur) ph_ld ^= 1u;
  ok = __syncthreads_and(ok) != 0;
  // warp roles: key path (the first 4 TPT warps) or value path; in each, warp w covers TMEM lane quarter
  // w % 4 (tokens 32 (w % 4) + lane) and, with two threads per row, column half (w % 8) / 4
  const bool kpath = warp < 4 * TPT;
  const int pw = warp % (4 * TPT), q4 = pw & 3, half = TPT == 2 ? (pw >> 2) : 0;
  const int t = 32 * q4 + lane;
  float* xs = reinterpret_cast<float*>(sm + Lq::kX);                  // [2 halves][128] partial |y'|^2
  float* xr = xs + 256;                                               // [2][128] partial |r|^2
  uint32_t* xw = reinterpret_cast<uint32_t*>(sm + Lq::kX + 2048);     // [4 MB][128] half-1 index words
  uint32_t* xg = reinterpret_cast<uint32_t*>(sm + Lq::kX + 8192);     // [4][128] half-1 sign words
  const PageLayout pl = page_layout(D, lv.vb, KB);
  // Writes key word cw of plane p for token t (column-half-0 threads, every lane of the warp), from both
  // column halves' bits (kbit_loc): at head_dim 128 one word per (token, plane, c); at head_dim 64 a word also
  // holds the odd 16-token tile of the token's 32-token group 8 bit positions up (lane ^ 16).
  auto put_word = [&](uint8_t* page, int p, int cw, uint32_t w) {
    uint32_t* kw = reinterpret_cast<uint32_t*>(page + pl.kbits_off);
    const int g = t & 7, r = (t >> 3) & 1;
    if constexpr (D == 128) {
      if (page) kw[(((t >> 4) * KB + p) * 32 + 4 * g + cw) * 2 + r] = w;
    } else {
      const uint32_t wo = __shfl_xor_sync(0xffffffffu, w, 16);
      if (page && ((t >> 4) & 1) == 0) kw[(((t >> 5) * KB + p) * 32 + 4 * g + cw) * 2 + r] = w | (wo << 8);
    }
  };
  uint8_t* prev_page = nullptr;  // page whose QJL signs are still to be written (its MMAs are in flight)
  bool prev = false;
  // Wait for the projection of the page in TMEM half `hb` (value warps); false if the wait gave up.
  auto qjl_wait = [&](uint32_t hb) -> bool {
    const bool w_ok = mbar_wait(bar_qjl2(hb), (ph_qjl >> hb) & 1u);
    if (tid == VL && w_ok) ++done[qjl_idx(hb)];
    ph_qjl ^= 1u << hb;
    return w_ok;
  };
  // QJL signs of the page in TMEM half `hb` (value warps, after qjl_wait): threshold z = S r, write the
  // sign plane.
  auto qjl_signs = [&](uint32_t hb, uint8_t* page) {
    tc_fence_after();
    const uint32_t prow = tmem + TH * hb + ((uint32_t)(32 * q4) << 16);
    uint32_t wsg[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int cc = 0; cc < HC / 32; ++cc) {
      uint32_t z[32];
      tmem_ld32(prow + HC * half + 32 * cc, z);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int jl = 32 * cc + i;
        const int cw = (jl >> 1) & 3, bit = 2 * (jl >> 4) + ((jl >> 3) & 1) + 16 * (jl & 1);
        wsg[cw] |= (__uint_as_float(z[i]) >= 0.f) ? (1u << bit) : 0u;
      }
    }
    if (half) {
#pragma unroll
      for (int cw = 0; cw < 4; ++cw) xg[cw * 128 + t] = wsg[cw] << PS;
    }
    tc_fence_before();
    named_barrier(2, HT);  // every value thread has read z (the half may be rotated into next)
    if constexpr (D == 128) {
      if (!half && page) {
        uint32_t* kw = reinterpret_cast<uint32_t*>(page + pl.kbits_off);
        const int ktile = t >> 4, kg = t & 7, kr = (t >> 3) & 1;
#pragma unroll
        for (int cw = 0; cw < 4; ++cw)
          kw[((ktile * KB + MB) * 32 + 4 * kg + cw) * 2 + kr] = wsg[cw] | (TPT == 2 ? xg[cw * 128 + t] : 0u);
      }
    } else if (!half) {
#pragma unroll
      for (int cw = 0; cw < 4; ++cw) put_word(page, MB, cw, wsg[cw] | (TPT == 2 ? xg[cw * 128 + t] : 0u));
    }
  };
  while (ok && cur < ntasks) {
    const int cslot = slot, chead = h, cpg = pg;
    const int nxt = bulk_next(a, cur + gridDim.x, ntasks, pages_per_row, rc, b, h, slot, L, Np, pg);
    const bool rot_ok = mbar_wait(bar_rot + bufi, (ph_rot >> bufi) & 1u);
    if (tid == 0 && rot_ok) ++done[4 + bufi];
    ok = __syncthreads_and(rot_ok) != 0;
    ph_rot ^= 1u << bufi;
    if (!ok) break;
    tc_fence_after();
    uint8_t* page = page_addr(lv, cslot, chead, cpg);
    const bool wr = page != nullptr;  // paged cache without a block for this page: code it, write nothing
    if (!wr && tid == 0) set_status(lv.status, TQ_DEV_ERR_BLOCK);
    const uint32_t lrow = tmem + TH * bufi + ((uint32_t)(32 * q4) << 16);
    bool ok_p = true;
    if (kpath) {
      // ---- keys, TPT threads per token (HC coordinates each): |y'|, y = y' / |y'|, index, residual ----
      float ss4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int cc = 0; cc < HC / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(lrow + HC * half + 32 * cc, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) ss4[i & 3] = fmaf(__uint_as_float(v[i]), __uint_as_float(v[i]), ss4[i & 3]);
      }
      const float ssum = (ss4[0] + ss4[1]) + (ss4[2] + ss4[3]);
      float nrot;  // = sqrt(d) |k|
      if constexpr (TPT == 2) {
        xs[half * 128 + t] = ssum;
        named_barrier(1, HT);
        nrot = sqrtf(xs[t] + xs[128 + t]);
      } else {
        nrot = sqrtf(ssum);
      }
      const float scale = nrot > 0.f ? 1.0f / nrot : 0.f;
      // The index of y = v / nrot (v = the rotated coordinate before normalisation) is decided as v > t nrot
      // for each boundary t (a zero vector compares v = 0 with t itself: y = 0), and the residual is
      // y - c = fma(v, 1 / nrot, -c).
      constexpr int NL = 1 << MB;  // Lloyd-Max levels
      float ncent[NL], bnd[NL - 1];
#pragma unroll
      for (int i = 0; i < NL; ++i) ncent[i] = -lv.cb[kCbCent + i];
#pragma unroll
      for (int i = 0; i < NL - 1; ++i) bnd[i] = nrot > 0.f ? lv.cb[kCbBnd + i] * nrot : lv.cb[kCbBnd + i];
      uint32_t wix[MB][4];  // index planes, highest bit first
#pragma unroll
      for (int p = 0; p < MB; ++p) wix[p][0] = wix[p][1] = wix[p][2] = wix[p][3] = 0u;
      float rr4[4] = {0.f, 0.f, 0.f, 0.f};
      // a whole row of 3-bit indices is coded in a rolled loop over its 32-column chunks (the unrolled
      // body outgrows the instruction cache); the chunk's bits are then 4 cc positions up
      constexpr int KCU = (TPT == 1 && MB == 3) ? 1 : HC / 32;
#pragma unroll KCU
      for (int cc = 0; cc < HC / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(lrow + HC * half + 32 * cc, v);
        uint32_t cwx[MB][4];  // the rolled loop: this chunk's index bits
#pragma unroll
        for (int p = 0; p < MB; ++p) cwx[p][0] = cwx[p][1] = cwx[p][2] = cwx[p][3] = 0u;
        (void)cwx;
#pragma unroll
        for (int oc = 0; oc < 4; ++oc) {  // 8 coordinates = one 16-byte chunk of the A rows
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            float res2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int i = 8 * oc + 2 * e2 + e;  // coordinate HC half + 32 cc + i
              const float vv = __uint_as_float(v[i]);
              // index = #{boundaries below y}, by binary search over the sorted (scaled) boundaries
              bool ib[MB];
              float ncv;
              if constexpr (MB == 2) {
                ib[0] = vv > bnd[1];
                ib[1] = vv > (ib[0] ? bnd[2] : bnd[0]);
                ncv = ib[0] ? (ib[1] ? ncent[3] : ncent[2]) : (ib[1] ? ncent[1] : ncent[0]);
              } else {
                ib[0] = vv > bnd[3];
                ib[1] = vv > (ib[0] ? bnd[5] : bnd[1]);
                ib[2] = vv > (ib[0] ? (ib[1] ? bnd[6] : bnd[4]) : (ib[1] ? bnd[2] : bnd[0]));
                ncv = ib[0] ? (ib[1] ? (ib[2] ? ncent[7] : ncent[6]) : (ib[2] ? ncent[5] : ncent[4]))
                            : (ib[1] ? (ib[2] ? ncent[3] : ncent[2]) : (ib[2] ? ncent[1] : ncent[0]));
              }
              const float res = fmaf(vv, scale, ncv);
              rr4[i & 3] = fmaf(res, res, rr4[i & 3]);
              res2[e] = res;
              // bit of coordinate j = HC half + 32 cc + i: word (j >> 1) & 3, bit 2 (j >> 4) + ((j >> 3) & 1) +
              // 16 (j & 1); 32 cc adds 4 cc to it and HC half adds PS = D / 16
              const int cw = (i >> 1) & 3, bit = 2 * (i >> 4) + ((i >> 3) & 1) + 16 * (i & 1);
              if constexpr (KCU == 1) {
#pragma unroll
                for (int p = 0; p < MB; ++p) cwx[p][cw] |= ib[p] ? (1u << bit) : 0u;
              } else {
#pragma unroll
                for (int p = 0; p < MB; ++p) wix[p][cw] |= ib[p] ? (1u << (bit + 4 * cc)) : 0u;
              }
            }
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(res2[0], res2[1]);
            const float2 hf2 = __bfloat1622float2(h2);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(res2[0] - hf2.x, res2[1] - hf2.y);
            hi[e2] = *reinterpret_cast<const uint32_t*>(&h2);
            lo[e2] = *reinterpret_cast<const uint32_t*>(&l2);
          }
          const uint32_t off = sw128_offset(t, HC * half + 32 * cc + 8 * oc);
          *reinterpret_cast<uint4*>(sm + Lq::kBuf + bufi * Lq::kBufBytes + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(sm + Lq::kBuf + bufi * Lq::kBufBytes + Lq::kTile + off) =
              make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        if constexpr (KCU == 1) {
#pragma unroll
          for (int p = 0; p < MB; ++p)
#pragma unroll
            for (int cw = 0; cw < 4; ++cw) wix[p][cw] |= cwx[p][cw] << (4 * cc);
        }
      }
      const float rsum = (rr4[0] + rr4[1]) + (rr4[2] + rr4[3]);
      if constexpr (TPT == 2) xr[half * 128 + t] = rsum;
      if (half) {
#pragma unroll
        for (int p = 0; p < MB; ++p)
#pragma unroll
          for (int cw = 0; cw < 4; ++cw) xw[(4 * p + cw) * 128 + t] = wix[p][cw] << PS;  // the upper half sits PS bit positions higher
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      tc_fence_before();
      named_barrier(1, HT);
      const uint32_t buf = buf0 + bufi * Lq::kBufBytes;
      if (tid == 0) {  // QJL: z = S r on the tensor cores (A = r hi, then r lo) over the consumed K columns
        tc_fence_after();
        const uint32_t ra = umma_desc_sw128_lo(buf), sa = umma_desc_sw128_lo(s_addr);
        constexpr int KS = D / 16;  // k steps per product
#pragma unroll
        for (int ks = 0; ks < 2 * KS; ++ks) {  // hi (ks < KS), then lo (+one tile); atoms of 16 KB, k steps of 32 B
          const uint32_t koff = ((ks % KS) >> 2) * 1024u + (ks & 3) * 2u;
          umma_bf16_lo(tmem + TH * bufi, ra + koff + (ks / KS) * (16u * D), sa + koff, kIdescBf16M128<D>, ks > 0);
        }
        umma_commit(bar_qjl2(bufi));  // waited on by the value warps in the next iteration (or after the loop)
        ++armed[qjl_idx(bufi)];
      }
      if (D == 128 ? (!half && wr) : !half) {  // index planes, n and gamma of token t
        if (wr) {
          const float n = nrot * rsqrtf((float)D);
          const float rr = TPT == 2 ? xr[t] + xr[128 + t] : rsum;
          const __half nh = __float2half_rn(fminf(n, 65504.f)), gh = __float2half_rn(sqrtf(rr));
          reinterpret_cast<uint32_t*>(page + pl.norms_off)[t] =
              (uint32_t)__half_as_ushort(nh) | ((uint32_t)__half_as_ushort(gh) << 16);
        }
        if constexpr (D == 128) {
          uint32_t* kw = reinterpret_cast<uint32_t*>(page + pl.kbits_off);
          const int tile = t >> 4, g = t & 7, r = (t >> 3) & 1;
#pragma unroll
          for (int p = 0; p < MB; ++p)
#pragma unroll
            for (int cw = 0; cw < 4; ++cw)
              kw[((tile * KB + p) * 32 + 4 * g + cw) * 2 + r] = wix[p][cw] | (TPT == 2 ? xw[(4 * p + cw) * 128 + t] : 0u);
        } else {
#pragma unroll
          for (int p = 0; p < MB; ++p)
#pragma unroll
            for (int cw = 0; cw < 4; ++cw)
              put_word(page, p, cw, wix[p][cw] | (TPT == 2 ? xw[(4 * p + cw) * 128 + t] : 0u));
        }
      }
    } else {
      // ---- the previous page's projection (it reads buffer bufi ^ 1); then the next page's copy starts
      // there at once (a TMA copy, by the value leader), and the signs of the previous page are written ----
      const bool nxt_tma = nxt < ntasks && pg * kPage >= L;  // b..pg describe the next page here
      if (prev) ok_p = qjl_wait(bufi ^ 1u);
      ld_skipped = nxt == a.fault_task;
      if (nxt_tma && ok_p)
        bulk_tc_load<D>(a, &tmk, &tmv, b, h, slot, L, Np, pg, sm + Lq::kBuf + (bufi ^ 1u) * Lq::kBufBytes,
                        bar_ld + (bufi ^ 1u), armed + 2 + (bufi ^ 1u), VL, 1, ld_skipped);
      if (prev) qjl_signs(bufi ^ 1u, prev_page);
      // a next page that starts in the ring is copied by all value threads (TMEM half bufi ^ 1 is free now)
      if (nxt < ntasks && !nxt_tma)
        bulk_tc_load<D>(a, &tmk, &tmv, b, h, slot, L, Np, pg, sm + Lq::kBuf + (bufi ^ 1u) * Lq::kBufBytes,
                        bar_ld + (bufi ^ 1u), armed + 2 + (bufi ^ 1u), VL, HT);
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // plain-copied rows -> tensor cores
      // ---- values, TPT threads per token (the D / (32 TPT) groups of 32 of its columns): fp16 scale,
      // mid-rise codes ----
      const int vhalf = 1 << (lv.vb - 1);
      const float inv_sqrt_d = rsqrtf((float)D);
      uint16_t* sw = reinterpret_cast<uint16_t*>(page + pl.vscale_off);
#pragma unroll 1
      for (int gg = 0; gg < D / (32 * TPT); ++gg) {
        const int grp = (D / (32 * TPT)) * half + gg;
        uint32_t v[32];
        tmem_ld32(lrow + D + 32 * grp, v);
        float x[32], am4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(v[i]) * inv_sqrt_d;
          am4[i & 3] = fmaxf(am4[i & 3], fabsf(x[i]));
        }
        const float am = fmaxf(fmaxf(am4[0], am4[1]), fmaxf(am4[2], am4[3]));
        const float s32 = fminf(__fdiv_rn(am, (float)vhalf - 0.5f), 65504.f);
        const __half sh = __float2half_rn(s32);
        const float sv = __half2float(sh);
        uint32_t cw[8];
        if (lv.vb == 2) {
          // code = clamp(floor(fl(x / s)), -2, 1) + 2 = [x >= -s] + [x >= 0] + [x >= s] for fp32 x and s > 0
          // (the rounded quotient's thresholds -(1 + 2^-24) and 1 - 2^-25 fall between s and its fp32
          // neighbours; see value_code), so no division is needed.
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint32_t w = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float xv = x[4 * k + e];
              const uint32_t code = (uint32_t)(xv >= -sv) + (uint32_t)(xv >= 0.f) + (uint32_t)(xv >= sv);
              w |= code << (8 * e);
            }
            cw[k] = sv > 0.f ? w : 0x02020202u;  // a zero group: every code 2
          }
        } else {
          // floor(x / s) with the quotient rounded as an IEEE division: x * (1/s) is within a few ulps of
          // it, so its floor is exact unless it lies within ~4 ulps of an integer; those (rare) elements
          // take the correctly rounded division.
          const float rcp = sv > 0.f ? __frcp_rn(sv) : 0.f;
          float fq[32];
          bool near = false;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float qv = x[i] * rcp;
            fq[i] = floorf(qv);
            const float fr = qv - fq[i], eps = fabsf(qv) * 4.8e-7f + 1e-30f;
            near |= (fr < eps) | (fr > 1.f - eps);
          }
          if (near && sv > 0.f) {
#pragma unroll
            for (int i = 0; i < 32; ++i) fq[i] = floorf(__fdiv_rn(x[i], sv));
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint32_t w = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int code = sv > 0.f ? (int)fminf(fmaxf(fq[4 * k + e], (float)-vhalf), (float)(vhalf - 1)) + vhalf : vhalf;
              w |= (uint32_t)code << (8 * e);
            }
            cw[k] = w;
          }
        }
        // vcode row t holds its 16-byte chunk k at chunk k ^ vsw(t) (conflict-free row writes)
        *reinterpret_cast<uint4*>(vcode + t * D + (((2 * grp) ^ vsw<D>(t)) << 4)) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        *reinterpret_cast<uint4*>(vcode + t * D + (((2 * grp + 1) ^ vsw<D>(t)) << 4)) =
            make_uint4(cw[4], cw[5], cw[6], cw[7]);
        if (wr) sw[vscale_idx(D, t, grp)] = __half_as_ushort(sh);
      }
      tc_fence_before();
      named_barrier(2, HT);  // value codes staged; V columns of this half read; next page's rows copied
      if (tid == VL && nxt < ntasks) {  // rotation of the next page into TMEM half bufi ^ 1
        tc_fence_after();
        bool landed = true;
        if (nxt_tma) {
          landed = mbar_wait(bar_ld + (bufi ^ 1u), (ph_ld >> (bufi ^ 1u)) & 1u, ld_skipped ? a.fault_polls : kWaitPolls);
          if (landed) ++done[2 + (bufi ^ 1u)];
          else set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
        }
        if (landed)
          bulk_tc_rotate<D>(tmem + TH * (bufi ^ 1u), buf0 + (bufi ^ 1u) * Lq::kBufBytes, hd_addr, bar_rot + (bufi ^ 1u),
                         armed + 4 + (bufi ^ 1u));
        else ok_p = false;
      }
      if (nxt_tma) ph_ld ^= 1u << (bufi ^ 1u);
      // ---- pack the value codes (fragment-major layout) ----
      const int vt = tid - VL;
      uint32_t* vw = reinterpret_cast<uint32_t*>(page + pl.vbits_off);
      if (lv.vb == 2) {
        for (int w = vt; w < 4 * (D / 16) * 32; w += HT) {
          const int ln = w & 31, mt = (w >> 5) % (D / 16), blk = w / (32 * (D / 16));
          const int g = ln >> 2, c = ln & 3;
          uint32_t word = 0;
#pragma unroll
          for (int kap = 0; kap < 2; ++kap)
#pragma unroll
            for (int rg = 0; rg < 4; ++rg)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int tt = 32 * blk + 16 * kap + 8 * (rg >> 1) + 2 * c + e;
                word |= (uint32_t)vcode[tt * D + ((mt ^ vsw<D>(tt)) << 4) + 8 * (rg & 1) + g] << (16 * e + 2 * vfield2(kap, rg));
              }
          if (wr) vw[w] = word;
        }
      } else {
        for (int w = vt; w < 4 * (D / 16) * 32 * 2; w += HT) {
          const int kap = w & 1, ln = (w >> 1) & 31, mt = (w >> 6) % (D / 16), blk = w / (64 * (D / 16));
          const int g = ln >> 2, c = ln & 3;
          uint32_t word = 0;
#pragma unroll
          for (int rg = 0; rg < 4; ++rg)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int tt = 32 * blk + 16 * kap + 8 * (rg >> 1) + 2 * c + e;
              word |= (uint32_t)vcode[tt * D + ((mt ^ vsw<D>(tt)) << 4) + 8 * (rg & 1) + g] << (16 * e + 4 * vfield4(rg));
            }
          if (wr) vw[w] = word;
        }
      }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok_p) != 0;  // the page is done; its buffer, vcode and exchange may be reused
    tc_fence_after();
    prev = true;
    prev_page = page;
    cur = nxt;
    bufi ^= 1u;
  }
  // the last page's QJL signs (its projection was issued in the final iteration)
  if (ok && prev && !kpath) {
    if (qjl_wait(bufi ^ 1u)) qjl_signs(bufi ^ 1u, prev_page);
    else ok = false;
  }
  if (!ok && (tid == 0 || tid == VL)) set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();  // every count is final
  // copies or MMAs still pending after a failed wait are waited for before shared memory and TMEM are
  // given up; a no-op after a run without one
  if (tid == 0 && !bulk_drain(bar_tab, 8, 6, armed, done)) set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
  __syncthreads();
  tc_fence_after();
  if (warp == 0)  // the 4 D columns allocated above
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "n"(4 * D) : "memory");
}

// Ring rows of a bulk append: the tokens past the last full page, [batch][pos][Hkv][K|V][d] items of
// 4 elements, spread over gridDim.y blocks per row. It reads the state before k_ring_update writes it.
__global__ void __launch_bounds__(256) k_ring_rows(AppendArgs a) {
  const int b = blockIdx.x;
  pdl_wait();  // the quantise launch has read the old ring and state
  const LayerView& lv = a.lv;
  const int slot = a.seq_ids[b];
  if (slot >= 0 && slot < lv.max_seqs) {
    const int L = lv.state[2 * slot];
    const int nn = new_count(a, b);
    const int L2 = L + nn;
    if (nn >= 0 && nn <= a.max_new && L2 <= lv.max_ctx) {
      const int Np2 = L2 > 0 ? kPage * ((L2 - 1) / kPage) : 0;
      const int p0 = max(L, Np2);
      const int d = lv.d, q4 = d / 4;
      const int n_items = (L2 - p0) * lv.Hkv * 2 * q4;  // (pos, head, which, quad)
      for (int it = blockIdx.y * blockDim.x + threadIdx.x; it < n_items; it += gridDim.y * blockDim.x) {
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
    }
  }
  __syncthreads();
  pdl_launch();
}

// Sequence state after an append (a.flush = 0, after k_ring_rows) or a ring flush (a.flush = 1).
// Dependents (the decode of this layer) are released only after the state is written: they read the
// sequence state before their own griddepcontrol.wait to start fetching pages early.
__global__ void __launch_bounds__(32) k_ring_update(AppendArgs a) {
  const int b = blockIdx.x;
  pdl_wait();  // the ring rows are written and the quantise launch has read the old state
  const LayerView& lv = a.lv;
  const int slot = a.seq_ids[b];
  if (threadIdx.x == 0 && slot >= 0 && slot < lv.max_seqs) {
    const int L = lv.state[2 * slot], F = lv.state[2 * slot + 1];
    const int Np = L > 0 ? kPage * ((L - 1) / kPage) : 0;
    if (a.flush) {
      lv.state[2 * slot + 1] = L - Np;
    } else {
      const int nn = new_count(a, b);
      const int L2 = L + nn;
      if (nn >= 0 && nn <= a.max_new && L2 <= lv.max_ctx) {
        const int Np2 = L2 > 0 ? kPage * ((L2 - 1) / kPage) : 0;
        lv.state[2 * slot] = L2;
        lv.state[2 * slot + 1] = Np2 > Np ? 0 : F;
      }
    }
    __threadfence();
  }
  __syncwarp();
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
  return quantize_smem_bytes_d<D>();
}

template <int D, int KB>
cudaError_t launch_quantize_dk(const AppendArgs& a, int batch, int pages, cudaStream_t s) {
  const size_t smem = quantize_smem_bytes<D>();
  static bool attr_set = false;  // set once, outside any stream capture that follows
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_quantize_pages<D, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (pages > 65535 / 4) return cudaErrorInvalidValue;  // grid z holds four 32-token CTAs per page
  dim3 grid(batch, a.lv.Hkv, 4 * pages);
  return launch_pdl(k_quantize_pages<D, KB>, grid, dim3(kQThreads), smem, s, a);
}

template <int D, int KB>
cudaError_t launch_append_small_dk(const AppendArgs& a, int batch, cudaStream_t s) {
  const size_t smem = quantize_smem_bytes<D>();
  static bool attr_set = false;  // set once, outside any stream capture that follows
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_append_small<D, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(k_append_small<D, KB>, dim3(batch, a.lv.Hkv, 4), dim3(kQThreads), smem, s, a);
}

cudaError_t launch_quantize(const AppendArgs& a, int batch, int pages, cudaStream_t s) {
  const bool k4 = a.lv.kb == 4;
  if (a.lv.d == 64) return k4 ? launch_quantize_dk<64, 4>(a, batch, pages, s) : launch_quantize_dk<64, 3>(a, batch, pages, s);
  if (a.lv.d == 128)
    return k4 ? launch_quantize_dk<128, 4>(a, batch, pages, s) : launch_quantize_dk<128, 3>(a, batch, pages, s);
  return k4 ? launch_quantize_dk<256, 4>(a, batch, pages, s) : launch_quantize_dk<256, 3>(a, batch, pages, s);
}

cudaError_t launch_append_small(const AppendArgs& a, int batch, cudaStream_t s) {
  const bool k4 = a.lv.kb == 4;
  if (a.lv.d == 64) return k4 ? launch_append_small_dk<64, 4>(a, batch, s) : launch_append_small_dk<64, 3>(a, batch, s);
  if (a.lv.d == 128) return k4 ? launch_append_small_dk<128, 4>(a, batch, s) : launch_append_small_dk<128, 3>(a, batch, s);
  return k4 ? launch_append_small_dk<256, 4>(a, batch, s) : launch_append_small_dk<256, 3>(a, batch, s);
}

template <int D, int KB>
cudaError_t launch_quantize_bulk_tc_k(const AppendArgs& a, int batch, int pages, int sms, cudaStream_t s) {
  // head_dim 64: a thread per token row and two CTAs per SM (101.5 KB of shared memory and 256 TMEM columns each)
  constexpr int TPT = D == 64 ? 1 : 2;
  constexpr size_t smem = QbLayout<D>::kSmem;
  static bool attr_set = false;  // set once, outside any stream capture that follows
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(k_quantize_bulk_tc<D, KB, TPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (TPT == 1) {  // the whole shared-memory carve-out, so that two CTAs fit on an SM
      e = cudaFuncSetAttribute(k_quantize_bulk_tc<D, KB, TPT>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return e;
    }
    attr_set = true;
  }
  const int ntasks = batch * a.lv.Hkv * pages;
  const int grid = std::max(1, std::min(ntasks, sms * (TPT == 1 ? 2 : 1)));
  CUtensorMap tmk, tmv;
  cudaError_t e = bulk_tensor_map(a.k, batch, a.max_new, a.lv.Hkv, D, &tmk);
  if (e == cudaSuccess) e = bulk_tensor_map(a.v, batch, a.max_new, a.lv.Hkv, D, &tmv);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_quantize_bulk_tc<D, KB, TPT>, dim3(grid), dim3(256 * TPT), smem, s, tmk, tmv, a, pages, batch);
}
// head_dim 64 or 128
cudaError_t launch_quantize_bulk_tc(const AppendArgs& a, int batch, int pages, int sms, cudaStream_t s) {
  const bool k4 = a.lv.kb == 4;
  if (a.lv.d == 64)
    return k4 ? launch_quantize_bulk_tc_k<64, 4>(a, batch, pages, sms, s) : launch_quantize_bulk_tc_k<64, 3>(a, batch, pages, sms, s);
  return k4 ? launch_quantize_bulk_tc_k<128, 4>(a, batch, pages, sms, s) : launch_quantize_bulk_tc_k<128, 3>(a, batch, pages, sms, s);
}

}  // namespace

// Tensor map of k or v ([batch][max_new][Hkv][d] bf16, d = 128 or 256) for 64 x 1 x 128 x 1 boxes
// (64 coordinates of 128 consecutive tokens of one head), 128-byte swizzle: the tcgen05 coders' page loads.
cudaError_t bulk_tensor_map(const void* base, int batch, int max_new, int hkv, int d, CUtensorMap* m) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t row = 2ull * d;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)hkv, (cuuint64_t)max_new, (cuuint64_t)batch};
  const cuuint64_t strides[3] = {row, (cuuint64_t)hkv * row, (cuuint64_t)max_new * hkv * row};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

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
  a.full = ctx->cfg.ring_size == 0;
  a.fault_task = g_qfault_task.load();
  a.fault_polls = (uint32_t)g_qfault_polls.load();
  if (max_new < kPage) return launch_append_small(a, batch, s);  // page on ring overflow + ring rows + state
  const int pages = (max_new + kPage - 1) / kPage;
  // the tcgen05 bulk coders serve bf16 appends at head_dim 64, 128 and 256 (key_bits 3 and 4); f32 inputs
  // use the CUDA-core coder
  const int sms = ctx->sm_count > 0 ? ctx->sm_count : 152;
  cudaError_t e = (a.lv.d <= 128 && dt == 0)   ? launch_quantize_bulk_tc(a, batch, pages, sms, s)
                  : (a.lv.d == 256 && dt == 0) ? launch_quantize_bulk256(a, batch, pages, sms, s)
                                               : launch_quantize(a, batch, pages, s);
  if (e != cudaSuccess) return e;
  // ring rows: up to 128 tokens x Hkv x (K, V) x d / 4 items per row, about 4 items per thread
  const int row_items = kPage * a.lv.Hkv * 2 * (a.lv.d / 4);
  e = launch_pdl(k_ring_rows, dim3(batch, (row_items + 1023) / 1024), dim3(256), 0, s, a);
  if (e == cudaSuccess) e = launch_pdl(k_ring_update, dim3(batch), dim3(32), 0, s, a);
  if (e != cudaSuccess || !a.full) return e;
  return launch_flush(ctx, layer, seq_ids, batch, s);  // full_tq: the partial page too
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
  a.full = 0;
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

extern "C" tq_status tq_debug_append_wait_fault(int task, int polls) {
  if (task < -1) return tq::set_error(TQ_ERR_INVALID_ARG, "task must be -1 (off) or >= 0");
  if (task >= 0 && (polls < 1 || polls > (int)tq::kWaitPolls))
    return tq::set_error(TQ_ERR_INVALID_ARG, "polls must be in [1, 2^22]");
  tq::g_qfault_polls.store(task >= 0 ? polls : 0);
  tq::g_qfault_task.store(task);
  return tq::set_error(TQ_OK, "");
}
