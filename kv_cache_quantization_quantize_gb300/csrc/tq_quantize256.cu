// Bulk quantise of head_dim 256 on tcgen05 tensor cores ([Guide] §二, the five steps of
// quantize-on-append, at the head_dim of [Guide] §六's fidelity table). One persistent CTA per SM
// walks its pages (128 tokens of one KV head) one at a time:
//   1. The bf16 K and V rows of the page arrive by eight TMA tensor copies (64 coordinates x 128
//      tokens each, 128-byte swizzle), or by plain loads when the page starts in the ring.
//   2. Rotation. The 256-point Sylvester Hadamard is H256 = [[H, H], [H, -H]] with H the 128-point
//      one, so with x = (x1, x2) and D = (D1, D2): H256 diag(D) x = (u1 + u2, u1 - u2) for
//      u1 = H diag(D1) x1 and u2 = H diag(D2) x2. The tensor cores form u1 and u2 of all 128 tokens
//      of K and of V (four M = N = K = 128 products against the +-1 tables, exact products, fp32
//      sums) into the 512 TMEM columns; the CUDA cores take the sum and the difference.
//   3. Warps 0-7 code the keys (two threads per token, each 64 columns of u1 and u2, that is 64
//      coordinates of each half): norm, Lloyd-Max index, residual, bf16 hi + lo split of the
//      residual written over the consumed K and V tiles. Warps 8-15 code the values (fp16 scale per
//      group of 32, mid-rise codes) and pack them into the page.
//   4. QJL: z = S r as N = 256 MMAs of the residual hi and lo against S, in four chunks of 64 columns
//      (K slices). Chunks 0 and 1 are copied into the H diag(D) tables' space as soon as the rotation
//      has read it (they land while the page is coded), chunk 2 into the staging space once the coding
//      is done, chunk 3 over chunk 0; z lands in the consumed key columns of TMEM. The tables are copied
//      back afterwards.
//   5. All warps threshold z into the sign plane while the next page's copy and the tables are in
//      flight.
#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "tq_quantize_common.cuh"
#include "tq_tcgen05.cuh"

namespace tq {
namespace {

constexpr int kQ2Threads = 512;        // warps 0-7 keys, 8-15 values; two warps (column halves) per token row
constexpr uint32_t kQ2HD = 0;          // H diag(D1) | H diag(D2): 2 x 32 KB, swizzled; S chunks 0/3 and 1 in the QJL
constexpr uint32_t kQ2X = 65536;       // K tile 64 KB (then residual hi) | V tile 64 KB (then residual lo)
constexpr uint32_t kQ2SB = kQ2X + 131072;  // 32 KB: exchange + value-code staging, then S chunk 2
constexpr uint32_t kQ2Bar = kQ2SB + 32768;  // mbarriers [8] (slot 7 holds the TMEM address), armed [8], done [8]
constexpr uint32_t kQ2Next = kQ2Bar + 128;  // the next page task, looked up by thread 0: [nxt, b, h, slot, L, Np, pg]
constexpr uint32_t kQ2End = kQ2Next + 32;
constexpr size_t kQ2Smem = kQ2End + 1024;  // + alignment slack for the 1024-byte swizzle atoms
// Inside SB while a page is coded: |u|^2 and |r|^2 partials, key index-word partials, value codes.
constexpr uint32_t kSbXs = 0, kSbXr = 1024, kSbXw = 2048, kSbVst = 16384;
// Barrier slots: the tables, the page copy, the rotation, S chunks in the table space halves 0 / 1 and in
// SB, the QJL MMA commits, the TMEM address.
constexpr int kB2Tab = 0, kB2Ld = 1, kB2Rot = 2, kB2S0 = 3, kB2S1 = 4, kB2S2 = 5, kB2M = 6, kB2Tmem = 7;
// kind::f16 instruction descriptor, bf16 operands, f32 accumulator, M = 128, N = 256.
constexpr uint32_t kIdescBf16M128N256 = (1u << 4) | (1u << 7) | (1u << 10) | ((256u >> 3) << 17) | ((128u >> 4) << 24);

static_assert(kQ2Smem <= 232448, "one CTA per SM: the 227 KB opt-in limit");
static_assert(kSbVst + 128 * 128 <= 32768, "value staging (4-bit codes) fits SB");
static_assert(kSbXw + 2 * 128 * 4 * 3 * 4 <= kSbVst, "key word partials (3 index planes) fit below the staging");

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// Loads page pg's K and V rows (bf16) into X: K tile at 0, V tile at 64 KB, each four 16 KB swizzle
// atoms of 64 coordinates (element (t, j) at sw128_offset(t, j)). Pages made of new input only are
// fetched by eight TMA tensor copies that complete on `bar` (returns true; thread 0 issues them and
// counts the arming in *armed). Pages that start in the ring are copied by all threads with plain loads.
// skip (test hook): a TMA copy is not issued at all (no expected bytes either), so its wait gives up.
__device__ __forceinline__ bool bulk256_load(const AppendArgs& a, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                             int b, int h, int slot, int L, int Np, int pg, uint8_t* x,
                                             uint64_t* bar, uint32_t* armed, bool skip) {
  constexpr int D = 256;
  const int tid = threadIdx.x;
  if (pg * kPage >= L) {
    if (tid == 0 && !skip) {
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      mbar_expect_tx(bar, 8u * 16384u);
      ++*armed;
      const int z = pg * kPage - L;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const CUtensorMap* m = i < 4 ? tmk : tmv;
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(
                smem_u32(x + i * 16384)),
            "l"(reinterpret_cast<uint64_t>(m)), "r"(64 * (i & 3)), "r"(h), "r"(z), "r"(b), "r"(smem_u32(bar))
            : "memory");
      }
    }
    return true;
  }
  for (int q = tid; q < 2 * kPage * (D / 8); q += kQ2Threads) {
    const int which = q >> 12, t = (q >> 5) & 127, c = q & 31;
    const int pos = pg * kPage + t;
    const uint16_t* src;
    if (pos < L) {
      src = a.lv.ring + ((((size_t)slot * a.lv.Hkv + h) * 2 + which) * kPage + (pos - Np)) * D;
    } else {
      src = static_cast<const uint16_t*>(which ? a.v : a.k) + (((size_t)b * a.max_new + (pos - L)) * a.lv.Hkv + h) * D;
    }
    *reinterpret_cast<uint4*>(x + which * 65536u + sw128_offset(t, 8 * c)) = *reinterpret_cast<const uint4*>(src + 8 * c);
  }
  return false;
}

// Prefetch of page pg's K and V rows (new input only) into L2, by the calling thread: the page copy
// that follows the next projection then reads L2 instead of HBM.
__device__ __forceinline__ void bulk256_prefetch(const CUtensorMap* tmk, const CUtensorMap* tmv, int b, int h, int L,
                                                 int pg) {
  const int z = pg * kPage - L;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(i < 4 ? tmk : tmv)),
                 "r"(64 * (i & 3)), "r"(h), "r"(z), "r"(b)
                 : "memory");
}

// Rotation products of the page in X (thread 0): TMEM columns [0, 128) = u1 of K, [128, 256) = u2 of K,
// [256, 384) = u1 of V, [384, 512) = u2 of V, with u_i[t][n] = sum_j x_i[t][j] (H diag(D_i))[n][j].
__device__ __forceinline__ void bulk256_rotate(uint32_t tmem, uint32_t x_addr, uint32_t hd_addr, uint64_t* bar,
                                               uint32_t* armed) {
  tc_fence_after();
  const uint32_t xa = umma_desc_sw128_lo(x_addr), hb = umma_desc_sw128_lo(hd_addr);
#pragma unroll
  for (int part = 0; part < 4; ++part) {
    // descriptor units of 16 bytes: V tile +4096, second 128 coordinates +2048, atom +1024, k step +2
    const uint32_t a0 = xa + (part >> 1) * 4096u + (part & 1) * 2048u, b0 = hb + (part & 1) * 2048u;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t koff = (ks >> 2) * 1024u + (ks & 3) * 2u;
      umma_bf16_lo(tmem + 128u * part, a0 + koff, b0 + koff, kIdescBf16M128N128, ks > 0);
    }
  }
  umma_commit(bar);
  ++*armed;
}

// Copy of S chunk q (columns [64q, 64q + 64) of all 256 rows: the table's 32 KB atom q) to dst,
// completing on bar.
__device__ __forceinline__ void bulk256_s_chunk(uint8_t* dst, const uint8_t* s_sw, int q, uint64_t* bar,
                                                uint32_t* armed) {
  mbar_expect_tx(bar, 32768u);
  ++*armed;
  bulk_g2s(dst, s_sw + (size_t)q * 32768, 32768u, bar);
}

// Per-barrier parity bits of the next waits, and the bounded wait that counts completions in done[].
struct Phases {
  uint32_t bits = 0;
  __device__ __forceinline__ bool wait(uint64_t* bars, int i, uint32_t* done, uint32_t polls = kWaitPolls) {
    if (!mbar_wait(bars + i, (bits >> i) & 1u, polls)) return false;
    ++done[i];
    bits ^= 1u << i;
    return true;
  }
};

// QJL projection of the page whose residual sits in X (hi at 0, lo at 64 KB; row t = token, column j =
// coordinate j), by thread 0: z[t][i] = sum_j (hi + lo)[t][j] S[i][j] into TMEM columns [0, 256), as
// N = 256 MMAs over the K slices j in [64q, 64q + 64) (chunk q of S). Chunks 0 and 1 were copied into the
// table space (halves 0 and 1) after the rotation; chunk 2 goes to SB now, chunk 3 into half 0 once chunk
// 0's MMAs have completed. Returns false if a wait gives up.
__device__ __forceinline__ bool bulk256_qjl(uint32_t tmem, uint32_t x_addr, uint8_t* hd, uint8_t* sb,
                                            const uint8_t* s_sw, uint64_t* bars, uint32_t* armed, uint32_t* done,
                                            Phases& ph) {
  bulk256_s_chunk(sb, s_sw, 2, bars + kB2S2, armed + kB2S2);
  const uint32_t xa = umma_desc_sw128_lo(x_addr);
  auto mmas = [&](int q, uint32_t chunk_addr) {
    tc_fence_after();
    const uint32_t bq = umma_desc_sw128_lo(chunk_addr);
#pragma unroll
    for (int hl = 0; hl < 2; ++hl)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // A: residual hi / lo (+4096), atom q (+1024 q), k step (+2 kk)
        umma_bf16_lo(tmem, xa + hl * 4096u + q * 1024u + kk * 2u, bq + kk * 2u, kIdescBf16M128N256,
                     (q | hl | kk) != 0);
  };
  const uint32_t hd_addr = smem_u32(hd);
  if (!ph.wait(bars, kB2S0, done)) return false;
  mmas(0, hd_addr);
  umma_commit(bars + kB2M);
  ++armed[kB2M];
  if (!ph.wait(bars, kB2S1, done)) return false;
  mmas(1, hd_addr + 32768u);
  if (!ph.wait(bars, kB2M, done)) return false;  // chunk 0's MMAs are done: half 0 takes chunk 3
  bulk256_s_chunk(hd, s_sw, 3, bars + kB2S0, armed + kB2S0);
  if (!ph.wait(bars, kB2S2, done)) return false;
  mmas(2, smem_u32(sb));
  if (!ph.wait(bars, kB2S0, done)) return false;
  mmas(3, hd_addr);
  umma_commit(bars + kB2M);
  ++armed[kB2M];
  return ph.wait(bars, kB2M, done);  // every MMA of the projection
}

// Index bit of column-local coordinate jl (0..63) of a thread's 64-column slice inside a key word of
// its 128-coordinate half (kbit_loc): word (jl >> 1) & 3, bit 2 (jl >> 4) + ((jl >> 3) & 1) + 16 (jl & 1);
// the slice of columns [64, 128) sits 8 bit positions higher.
__device__ __forceinline__ constexpr int kw_word(int jl) { return (jl >> 1) & 3; }
__device__ __forceinline__ constexpr int kw_bit(int jl) { return 2 * (jl >> 4) + ((jl >> 3) & 1) + 16 * (jl & 1); }

// Keys of the page (warps 0-7, thread (t, hp): columns [64 hp, 64 hp + 64) of u1 and u2, i.e.
// coordinates c and 128 + c for c in that range). Writes the residual hi / lo into X, the index planes
// and {n, gamma} into the page (when wr).
template <int KB>
__device__ __forceinline__ void bulk256_keys(const LayerView& lv, uint32_t lrow, int t, int hp, uint8_t* x, uint8_t* sb,
                                             uint8_t* page, bool wr) {
  constexpr int D = 256, MB = KB - 1;
  float* xs = reinterpret_cast<float*>(sb + kSbXs);      // [2][128] partial |u1|^2 + |u2|^2
  float* xr = reinterpret_cast<float*>(sb + kSbXr);      // [2][128] partial |r|^2
  uint32_t* xw = reinterpret_cast<uint32_t*>(sb + kSbXw);  // [half][4 MB][128] partner's index-word partials
  // ---- |y'|^2 = |u1 + u2|^2 + |u1 - u2|^2 = 2 (|u1|^2 + |u2|^2) ----
  float ss4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int sc = 0; sc < 4; ++sc) {
    uint32_t u1[16], u2[16];
    tmem_ld16(lrow + 64 * hp + 16 * sc, u1);
    tmem_ld16(lrow + 128 + 64 * hp + 16 * sc, u2);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      ss4[i & 3] = fmaf(__uint_as_float(u1[i]), __uint_as_float(u1[i]), ss4[i & 3]);
      ss4[i & 3] = fmaf(__uint_as_float(u2[i]), __uint_as_float(u2[i]), ss4[i & 3]);
    }
  }
  xs[hp * 128 + t] = (ss4[0] + ss4[1]) + (ss4[2] + ss4[3]);
  named_barrier(1, 256);
  const float nrot = sqrtf(2.f * (xs[t] + xs[128 + t]));  // = sqrt(d) |k|
  const float scale = nrot > 0.f ? 1.0f / nrot : 0.f;
  // The index of y = v / nrot (v = the rotated coordinate before normalisation) is decided as v > t nrot for
  // each boundary t (a zero vector compares v = 0 with t itself: y = 0), and the residual is
  // y - c = fma(v, 1 / nrot, -c).
  constexpr int NL = 1 << MB;
  float ncent[NL], bnd[NL - 1];
#pragma unroll
  for (int i = 0; i < NL; ++i) ncent[i] = -lv.cb[kCbCent + i];
#pragma unroll
  for (int i = 0; i < NL - 1; ++i) bnd[i] = nrot > 0.f ? lv.cb[kCbBnd + i] * nrot : lv.cb[kCbBnd + i];
  // The half 1 - hp is coded first and its index-word partials handed to the partner (which writes the
  // words of that half); the words of half hp stay in registers.
  uint32_t wix[MB][4];  // [plane, highest index bit first][word] of the half being coded
  float rr4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int hf = it ? hp : 1 - hp;  // hf 0: coordinate c = u1 + u2; hf 1: coordinate 128 + c = u1 - u2
    const float sgn = hf ? -1.f : 1.f;
#pragma unroll
    for (int p = 0; p < MB; ++p) wix[p][0] = wix[p][1] = wix[p][2] = wix[p][3] = 0u;
#pragma unroll
    for (int sc = 0; sc < 4; ++sc) {
      uint32_t u1[16], u2[16];
      tmem_ld16(lrow + 64 * hp + 16 * sc, u1);
      tmem_ld16(lrow + 128 + 64 * hp + 16 * sc, u2);
#pragma unroll
      for (int oc = 0; oc < 2; ++oc) {  // 8 coordinates = one 16-byte chunk of the A rows
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          float res2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = 8 * oc + 2 * e2 + e, jl = 16 * sc + i;
            const float vv = fmaf(sgn, __uint_as_float(u2[i]), __uint_as_float(u1[i]));
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
#pragma unroll
            for (int p = 0; p < MB; ++p) wix[p][kw_word(jl)] |= ib[p] ? (1u << kw_bit(jl)) : 0u;
          }
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(res2[0], res2[1]);
          const float2 hf2 = __bfloat1622float2(h2);
          const __nv_bfloat162 l2 = __floats2bfloat162_rn(res2[0] - hf2.x, res2[1] - hf2.y);
          hi[e2] = *reinterpret_cast<const uint32_t*>(&h2);
          lo[e2] = *reinterpret_cast<const uint32_t*>(&l2);
        }
        const uint32_t off = sw128_offset(t, 128 * hf + 64 * hp + 16 * sc + 8 * oc);
        *reinterpret_cast<uint4*>(x + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(x + 65536u + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    if (it == 0) {  // the partner writes the words of half 1 - hp: hand it ours
#pragma unroll
      for (int p = 0; p < MB; ++p)
#pragma unroll
        for (int cw = 0; cw < 4; ++cw) xw[((1 - hp) * 4 * MB + 4 * p + cw) * 128 + t] = wix[p][cw];
    }
  }
  xr[hp * 128 + t] = (rr4[0] + rr4[1]) + (rr4[2] + rr4[3]);
  named_barrier(1, 256);
  if (wr) {
    uint32_t* kw = reinterpret_cast<uint32_t*>(page + page_layout(D, lv.vb, KB).kbits_off);
    const int tile = t >> 4, g = t & 7, r = (t >> 3) & 1;
#pragma unroll
    for (int p = 0; p < MB; ++p)
#pragma unroll
      for (int cw = 0; cw < 4; ++cw) {
        const uint32_t own = wix[p][cw];
        const uint32_t other = xw[(hp * 4 * MB + 4 * p + cw) * 128 + t];
        kw[(((tile * KB + p) * 2 + hp) * 32 + 4 * g + cw) * 2 + r] = (own << (8 * hp)) | (other << (8 * (1 - hp)));
      }
    if (hp == 0) {  // n and gamma of token t
      const float n = nrot * 0.0625f;  // / sqrt(256)
      const float rr = xr[t] + xr[128 + t];
      const __half nh = __float2half_rn(fminf(n, 65504.f)), gh = __float2half_rn(sqrtf(rr));
      reinterpret_cast<uint32_t*>(page + page_layout(D, lv.vb, KB).norms_off)[t] =
          (uint32_t)__half_as_ushort(nh) | ((uint32_t)__half_as_ushort(gh) << 16);
    }
  }
}

// Mid-rise codes of one group of 32 rotated value coordinates x with fp16 scale sv, given as x16 = 16 x
// (exact: the 1 / sqrt(256) of the rotation is a power of two), packed by coordinate: vb 2: w[k] holds
// coordinates 16k..16k+15 at bits 2i (k < 2); vb 4: w[k] holds coordinates 8k..8k+7 at bits 4i (k < 4).
// A zero group (sv = 0) codes every coordinate as 2^(vb-1).
__device__ __forceinline__ void value_group_codes(const float (&x16)[32], float sv, int vb, uint32_t (&w)[4]) {
  if (vb == 2) {
    const float sv16 = sv * 16.f;  // exact
    // code = clamp(floor(fl(x / s)), -2, 1) + 2 = [x >= -s] + [x >= 0] + [x >= s] for fp32 x and s > 0 (the
    // rounded quotient's thresholds -(1 + 2^-24) and 1 - 2^-25 fall between s and its fp32 neighbours), so
    // no division is needed.
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      uint32_t acc = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float xv = x16[16 * k + i];
        const uint32_t code = (uint32_t)(xv >= -sv16) + (uint32_t)(xv >= 0.f) + (uint32_t)(xv >= sv16);
        acc |= code << (2 * i);
      }
      w[k] = sv > 0.f ? acc : 0xAAAAAAAAu;
    }
    w[2] = w[3] = 0u;
    return;
  }
  // floor(x / s) with the quotient rounded as an IEEE division: x * (1/s) is within a few ulps of it, so its
  // floor is exact unless it lies within ~4 ulps of an integer; those (rare) groups take the division.
  const float rcp16 = sv > 0.f ? __frcp_rn(sv) * 0.0625f : 0.f;  // x16 * rcp16 = x * (1 / s) exactly
  float fq[32];
  bool near = false;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float qv = x16[i] * rcp16;
    fq[i] = floorf(qv);
    const float fr = qv - fq[i], eps = fabsf(qv) * 4.8e-7f + 1e-30f;
    near |= (fr < eps) | (fr > 1.f - eps);
  }
  if (near && sv > 0.f) {
#pragma unroll
    for (int i = 0; i < 32; ++i) fq[i] = floorf(__fdiv_rn(x16[i] * 0.0625f, sv));
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t acc = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int code = sv > 0.f ? (int)fminf(fmaxf(fq[8 * k + i], -8.f), 7.f) + 8 : 8;
      acc |= (uint32_t)code << (4 * i);
    }
    w[k] = acc;
  }
}

// Values of the page (warps 8-15, thread (t, hp): columns [64 hp, 64 hp + 64) of u1 and u2 of V, i.e.
// the groups 2 hp, 2 hp + 1 (u1 + u2) and 4 + 2 hp, 5 + 2 hp (u1 - u2)). Scales go to the page from
// registers; codes are staged in SB by token (vb 2: 64 B per token, group g in the 8-byte slot
// g ^ ((t >> 1) & 7); vb 4: 128 B per token, group g in the 16-byte slot g ^ (t & 7)) and then packed
// into the fragment-major value words (vcode_loc) by the 256 value threads.
__device__ __forceinline__ void bulk256_values(const LayerView& lv, uint32_t lrow, int t, int hp, int vt, uint8_t* sb,
                                               uint8_t* page, bool wr, const PageLayout& pl) {
  constexpr int D = 256;
  const int vb = lv.vb, vhalf = 1 << (vb - 1);
  uint8_t* vst = sb + kSbVst;
  uint16_t* sw = reinterpret_cast<uint16_t*>(page + pl.vscale_off);
#pragma unroll 1
  for (int cc = 0; cc < 2; ++cc) {
    uint32_t u1[32], u2[32];
    tmem_ld32(lrow + 256 + 64 * hp + 32 * cc, u1);
    tmem_ld32(lrow + 384 + 64 * hp + 32 * cc, u2);
    float xs2[2][32];  // [0] = u1 + u2, [1] = u1 - u2: 16 times the rotated coordinates, formed in place
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float a1 = __uint_as_float(u1[i]), a2 = __uint_as_float(u2[i]);
      xs2[0][i] = a1 + a2;
      xs2[1][i] = a1 - a2;
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int grp = 4 * hf + 2 * hp + cc;
      const float(&x)[32] = xs2[hf];
      float am4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 32; ++i) am4[i & 3] = fmaxf(am4[i & 3], fabsf(x[i]));
      const float am = fmaxf(fmaxf(am4[0], am4[1]), fmaxf(am4[2], am4[3])) * 0.0625f;  // exact
      const float s32 = fminf(__fdiv_rn(am, (float)vhalf - 0.5f), 65504.f);
      const __half sh = __float2half_rn(s32);
      uint32_t w[4];
      value_group_codes(x, __half2float(sh), vb, w);
      if (vb == 2) {
        *reinterpret_cast<uint2*>(vst + 64 * t + 8 * (grp ^ ((t >> 1) & 7))) = make_uint2(w[0], w[1]);
      } else {
        *reinterpret_cast<uint4*>(vst + 128 * t + 16 * (grp ^ (t & 7))) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      if (wr) sw[vscale_idx(D, t, grp)] = __half_as_ushort(sh);
    }
  }
  named_barrier(2, 256);  // every token's codes are staged
  if (!wr) return;
  uint32_t* vw = reinterpret_cast<uint32_t*>(page + pl.vbits_off);
  // the lane field of the words w = vt + 256 k is fixed per thread: bits 0-4 of w (vb 2), 1-5 (vb 4)
  const int ln = vb == 2 ? (vt & 31) : ((vt >> 1) & 31), g = ln >> 2, c = ln & 3;
  if (vb == 2) {
    // word (blk, mt, lane 4g + c): tokens 32 blk + 16 kap + 8 hi + 2c + e, coordinates 16 mt + 8 rowhi + g;
    // both rowhi of a token sit in staged word mt (bits 2g and 2g + 16)
#pragma unroll 1
    for (int w = vt; w < 4 * (D / 16) * 32; w += 256) {
      const int mt = (w >> 5) & 15, blk = w >> 9;
      uint32_t word = 0;
#pragma unroll
      for (int kap = 0; kap < 2; ++kap)
#pragma unroll
        for (int hi = 0; hi < 2; ++hi)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tt = 32 * blk + 16 * kap + 8 * hi + 2 * c + e;
            const uint32_t sx =
                *reinterpret_cast<const uint32_t*>(vst + 64 * tt + 8 * ((mt >> 1) ^ ((tt >> 1) & 7)) + 4 * (mt & 1)) >> (2 * g);
            word |= (sx & 3u) << (16 * e + 2 * vfield2(kap, 2 * hi));
            word |= ((sx >> 16) & 3u) << (16 * e + 2 * vfield2(kap, 2 * hi + 1));
          }
      vw[w] = word;
    }
  } else {
    // word (blk, mt, lane, kap): tokens 32 blk + 16 kap + 8 hi + 2c + e, coordinates 16 mt + 8 rowhi + g;
    // the two rowhi of a token sit in staged words 2 mt and 2 mt + 1 (nibble g)
#pragma unroll 1
    for (int w = vt; w < 4 * (D / 16) * 32 * 2; w += 256) {
      const int kap = w & 1, mt = (w >> 6) & 15, blk = w >> 10;
      uint32_t word = 0;
#pragma unroll
      for (int hi = 0; hi < 2; ++hi)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tt = 32 * blk + 16 * kap + 8 * hi + 2 * c + e;
          const uint2 sx =
              *reinterpret_cast<const uint2*>(vst + 128 * tt + 16 * ((mt >> 1) ^ (tt & 7)) + 8 * (mt & 1));
          word |= ((sx.x >> (4 * g)) & 15u) << (16 * e + 4 * vfield4(2 * hi));
          word |= ((sx.y >> (4 * g)) & 15u) << (16 * e + 4 * vfield4(2 * hi + 1));
        }
      vw[w] = word;
    }
  }
}

// QJL signs of the page (all 16 warps; warp w: TMEM lane quarter w % 4, projections [64 qc, 64 qc + 64)
// with qc = w / 4, i.e. half qc / 2 of the sign plane, slice qc % 2). Slice-1 threads hand their partial
// words (8 bit positions up) to the slice-0 thread of the same token and half through SB, which writes
// them. Ends with a block barrier.
template <int KB>
__device__ __forceinline__ void bulk256_signs(uint32_t tmem, int warp, int lane, uint8_t* sb, uint8_t* page, bool wr,
                                              const PageLayout& pl) {
  const int q4 = warp & 3, qc = warp >> 2, half = qc >> 1, sl = qc & 1;
  const int t = 32 * q4 + lane;
  uint32_t* xg = reinterpret_cast<uint32_t*>(sb);  // [half][4][128]
  uint32_t wsg[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    uint32_t z[32];
    tmem_ld32(tmem + ((uint32_t)(32 * q4) << 16) + 64 * qc + 32 * cc, z);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int jl = 32 * cc + i;
      wsg[kw_word(jl)] |= (__uint_as_float(z[i]) >= 0.f) ? (1u << kw_bit(jl)) : 0u;
    }
  }
  if (sl) {
#pragma unroll
    for (int cw = 0; cw < 4; ++cw) xg[(half * 4 + cw) * 128 + t] = wsg[cw] << 8;
  }
  tc_fence_before();
  __syncthreads();
  if (!sl && wr) {
    constexpr int MB = KB - 1;
    uint32_t* kw = reinterpret_cast<uint32_t*>(page + pl.kbits_off);
    const int tile = t >> 4, g = t & 7, r = (t >> 3) & 1;
#pragma unroll
    for (int cw = 0; cw < 4; ++cw)
      kw[(((tile * KB + MB) * 2 + half) * 32 + 4 * g + cw) * 2 + r] = wsg[cw] | xg[(half * 4 + cw) * 128 + t];
  }
}

// KB = key bits: 3 (2-bit Lloyd-Max index + sign) or 4 (3-bit index + sign).
template <int KB>
__global__ void __launch_bounds__(kQ2Threads, 1)
    k_quantize_bulk256(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, AppendArgs a,
                       int pages_per_row, int batch) {
  constexpr int D = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* x = sm + kQ2X;
  uint8_t* sb = sm + kQ2SB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kQ2Bar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kB2Tmem);
  // phases armed on barrier i and seen complete by thread 0 (every barrier is armed and counted by it)
  uint32_t* armed = reinterpret_cast<uint32_t*>(bars + 8);
  uint32_t* done = armed + 8;
  const LayerView& lv = a.lv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_launch();
  if (tid == 0) {
    for (int i = 0; i < 16; ++i) armed[i] = 0u;  // armed[8], done[8]
    for (int i = 0; i < 7; ++i) mbar_init(bars + i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    mbar_expect_tx(bars + kB2Tab, 65536u);
    armed[kB2Tab] = 1u;
    bulk_g2s(sm + kQ2HD, lv.HD_sw, 32768u, bars + kB2Tab);
    bulk_g2s(sm + kQ2HD + 32768, reinterpret_cast<const uint8_t*>(lv.HD_sw) + 32768, 32768u, bars + kB2Tab);
  }
  if (warp == 0) {  // all 512 TMEM columns: [u1 K | u2 K | u1 V | u2 V], then z = S r over the key half
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(tslot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t hd_addr = smem_u32(sm + kQ2HD), x_addr = smem_u32(x);
  const int ntasks = batch * lv.Hkv * pages_per_row;
  const PageLayout pl = page_layout(D, lv.vb, KB);
  int b, h, slot, L, Np, pg;
  RowTask rc;  // this thread's cached row lookup
  int cur = bulk_next(a, blockIdx.x, ntasks, pages_per_row, rc, b, h, slot, L, Np, pg);
  bool ld_skipped = cur == a.fault_task;  // the wait-timeout test hook: this page's copy is not issued
  bool tma = cur < ntasks && bulk256_load(a, &tmk, &tmv, b, h, slot, L, Np, pg, x, bars + kB2Ld, armed + kB2Ld,
                                          ld_skipped);
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // plain-copied rows -> tensor cores
  __syncthreads();  // every plain-copied row is in X before thread 0 issues the rotation
  bool ok = true;
  Phases ph;            // thread 0: parities of the table, page-copy, S-chunk and MMA-commit barriers
  uint32_t ph_rot = 0;  // every thread waits for the rotation
  const bool kpath = warp < 8;
  const int q4 = warp & 3, hp = (warp >> 2) & 1;  // TMEM lane quarter, column slice
  const int t = 32 * q4 + lane;
  const uint32_t lrow = tmem + ((uint32_t)(32 * q4) << 16);
  while (ok && cur < ntasks) {
    uint8_t* page = page_addr(lv, slot, h, pg);
    // ---- rotation of the page in X, once its copy and the tables have landed ----
    if (tid == 0) {
      const bool landed =
          ph.wait(bars, kB2Tab, done) && (!tma || ph.wait(bars, kB2Ld, done, ld_skipped ? a.fault_polls : kWaitPolls));
      if (landed) bulk256_rotate(tmem, x_addr, hd_addr, bars + kB2Rot, armed + kB2Rot);
      else ok = false;
    }
    if (tid == 32) {  // the next task, while the rotation runs (its state loads are off every other path)
      int* nt = reinterpret_cast<int*>(sm + kQ2Next);
      int nb, nh, ns, nL, nNp, npg;
      const int nx = bulk_next(a, cur + gridDim.x, ntasks, pages_per_row, rc, nb, nh, ns, nL, nNp, npg, 32);
      if (nx < ntasks && npg * kPage >= nL) bulk256_prefetch(&tmk, &tmv, nb, nh, nL, npg);
      nt[0] = nx, nt[1] = nb, nt[2] = nh, nt[3] = ns, nt[4] = nL, nt[5] = nNp, nt[6] = npg;
    }
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    const bool rot_ok = mbar_wait(bars + kB2Rot, ph_rot);
    if (tid == 0 && rot_ok) {
      ++done[kB2Rot];
      // the tables are read: their space takes S chunks 0 and 1 while the page is coded
      bulk256_s_chunk(sm + kQ2HD, reinterpret_cast<const uint8_t*>(lv.S_sw), 0, bars + kB2S0, armed + kB2S0);
      bulk256_s_chunk(sm + kQ2HD + 32768, reinterpret_cast<const uint8_t*>(lv.S_sw), 1, bars + kB2S1, armed + kB2S1);
    }
    ph_rot ^= 1u;
    ok = __syncthreads_and(rot_ok) != 0;
    if (!ok) break;
    tc_fence_after();
    const bool wr = page != nullptr;  // paged cache without a block for this page: code it, write nothing
    if (!wr && tid == 0) set_status(lv.status, TQ_DEV_ERR_BLOCK);
    // ---- keys (warps 0-7) and values (warps 8-15) ----
    if (kpath) bulk256_keys<KB>(lv, lrow, t, hp, x, sb, page, wr);
    else bulk256_values(lv, lrow, t, hp, tid - 256, sb, page, wr, pl);
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // residual rows -> tensor cores; SB -> copies
    tc_fence_before();
    __syncthreads();  // X holds the residual, the key columns of TMEM are read, SB is free
    const int* nt = reinterpret_cast<const int*>(sm + kQ2Next);
    const int nxt = nt[0];
    b = nt[1], h = nt[2], slot = nt[3], L = nt[4], Np = nt[5], pg = nt[6];
    // ---- QJL projection (thread 0) ----
    if (tid == 0) {
      tc_fence_after();
      ok = bulk256_qjl(tmem, x_addr, sm + kQ2HD, sb, reinterpret_cast<const uint8_t*>(lv.S_sw), bars, armed, done, ph);
      if (ok && nxt < ntasks) {  // the tables back for the next page's rotation
        mbar_expect_tx(bars + kB2Tab, 65536u);
        ++armed[kB2Tab];
        bulk_g2s(sm + kQ2HD, lv.HD_sw, 32768u, bars + kB2Tab);
        bulk_g2s(sm + kQ2HD + 32768, reinterpret_cast<const uint8_t*>(lv.HD_sw) + 32768, 32768u, bars + kB2Tab);
      }
    }
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    tc_fence_after();
    // ---- the next page's copy (X is free: the projection has completed), then the signs ----
    ld_skipped = nxt == a.fault_task;
    tma = nxt < ntasks && bulk256_load(a, &tmk, &tmv, b, h, slot, L, Np, pg, x, bars + kB2Ld, armed + kB2Ld, ld_skipped);
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    bulk256_signs<KB>(tmem, warp, lane, sb, page, wr, pl);
    tc_fence_before();
    __syncthreads();  // SB and the z columns are read
    cur = nxt;
  }
  if (!ok && tid == 0) set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();  // every count is final
  // copies or MMAs still pending after a failed wait are waited for before shared memory and TMEM are
  // given up; a no-op after a run without one
  if (tid == 0 && !bulk_drain(bars, 8, kB2Tmem, armed, done)) set_status(lv.status, TQ_DEV_ERR_TIMEOUT);
  __syncthreads();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem) : "memory");
}

template <int KB>
cudaError_t launch_bulk256_k(const AppendArgs& a, int batch, int pages, int sms, cudaStream_t s) {
  static bool attr_set = false;  // set once, outside any stream capture that follows
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_quantize_bulk256<KB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQ2Smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int ntasks = batch * a.lv.Hkv * pages;
  const int grid = std::max(1, std::min(ntasks, sms));
  CUtensorMap tmk, tmv;
  cudaError_t e = bulk_tensor_map(a.k, batch, a.max_new, a.lv.Hkv, 256, &tmk);
  if (e == cudaSuccess) e = bulk_tensor_map(a.v, batch, a.max_new, a.lv.Hkv, 256, &tmv);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_quantize_bulk256<KB>, dim3(grid), dim3(kQ2Threads), kQ2Smem, s, tmk, tmv, a, pages, batch);
}

}  // namespace

cudaError_t launch_quantize_bulk256(const AppendArgs& a, int batch, int pages, int sms, cudaStream_t s) {
  return a.lv.kb == 4 ? launch_bulk256_k<4>(a, batch, pages, sms, s) : launch_bulk256_k<3>(a, batch, pages, sms, s);
}

}  // namespace tq
