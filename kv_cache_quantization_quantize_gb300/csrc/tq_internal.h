// Internal declarations of libtq: page layout, context, kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "tq.h"

#if defined(__CUDACC__)
#define TQ_HD __host__ __device__ __forceinline__
#else
#define TQ_HD inline
#endif

namespace tq {

// NVTX range named after the C-ABI call it covers (Nsight Systems timelines, ncu --nvtx filters). With
// no tool attached the push and pop are a load and a branch each.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kPage = 128;  // tokens per packed page = ring capacity ([Guide] §五.1 buffer_size=128)
constexpr int kMaxG = 4;    // query heads per KV head served by one decode CTA (GQA <= 4)

// ---------------------------------------------------------------------------------------------
// Packed page of 128 tokens of one KV head. The layout is fragment-major: the decode kernel's
// mma.sync operand registers are cut out of it with one LOP3 per 2 elements. Sections:
//   KBITS  [tile 8][plane kb][half d/128][lane 32][row 2] u32 (see kbit_loc), kb = key_bits planes:
//          planes 0 .. kb-2 = the Lloyd-Max index bits from the highest down, plane kb-1 = QJL sign
//          (1 = z >= 0).
//   NORMS  [token 128] {fp16 n, fp16 gamma}.
//   VBITS  2-bit: [block 4][m-tile d/16][lane 32] u32; 4-bit: [block 4][m-tile d/16][lane 32][2] u32.
//   VSCALE [token/2 64][group d/32][token&1 2] fp16 (pairs of consecutive tokens per group).
// Per token: K (kb*d/8 + 4 B) + V (d*vb/8 + d/16 B); d=128, K3/V2 -> 92 B, identical to the canonical
// record size. A page is therefore the canonical records in another order.
// ---------------------------------------------------------------------------------------------
struct PageLayout {
  int d, vb, kb;
  uint32_t kbits_off, norms_off, vbits_off, vscale_off, bytes;
};

TQ_HD PageLayout page_layout(int d, int vb, int kb) {
  PageLayout p;
  p.d = d;
  p.vb = vb;
  p.kb = kb;
  p.kbits_off = 0;
  p.norms_off = p.kbits_off + (uint32_t)kb * kPage * d / 8;
  p.vbits_off = p.norms_off + 4u * kPage;
  p.vscale_off = p.vbits_off + (uint32_t)kPage * d * vb / 8;
  p.bytes = p.vscale_off + 2u * kPage * (d / 32);
  return p;
}

// Location of the key bit of (token t, coordinate j, plane pi) in KBITS of a page with kb planes: u32
// word index and bit. KBITS is [tile 8][plane kb][half d/128][lane 32][row 2] u32. Tile = 16 tokens, row r = token bit 3,
// lane = 4g + c with g = token bits 0-2. Bit q + 16e of a word holds coordinate
// 128*half + 16s + 8sub + 2c + e, with pair index q = 2s + sub. Masking bits q and q + 16 of a word
// gives the f16 pair of m16n8k16 operand A (rows = tokens, k = coordinates). For q < 12 each half is
// exactly 2^(q-24) when set; pairs 12..15 are shifted down by 4 first.
// head_dim 64 has 4 pair indices per tile, so one word holds both tiles of a 32-token group: KBITS is
// [group 4][plane kb][lane 32][row 2] u32 and the odd tile sits 8 bit positions higher (the decoder
// shifts it down by 8 first).
TQ_HD void kbit_loc(int d, int kb, int t, int j, int pi, int& word, int& bit) {
  const int tile = t >> 4, g = t & 7, r = (t >> 3) & 1;
  const int half = j >> 7, jj = j & 127;
  const int s = jj >> 4, sub = (jj >> 3) & 1, c = (jj >> 1) & 3, e = jj & 1;
  if (d == 64) {
    word = (((tile >> 1) * kb + pi) * 32 + 4 * g + c) * 2 + r;
    bit = 2 * s + sub + 8 * (tile & 1) + 16 * e;
    return;
  }
  word = ((((tile * kb + pi) * (d >> 7) + half) * 32) + 4 * g + c) * 2 + r;
  bit = 2 * s + sub + 16 * e;
}
// Bit of plane pi in a per-coordinate key code (idx | sign << (kb - 1)): index bits from the highest
// down, then the sign.
TQ_HD int plane_bit(int code, int pi, int kb) { return (code >> (pi < kb - 1 ? kb - 2 - pi : kb - 1)) & 1; }

// Effective bit position (after the decoder's shift) of pair index q.
TQ_HD int kpair_pos(int q) { return q < 12 ? q : q - 4; }

// Field tables of the value words (see vcode_loc): which 2-bit (4-bit) field of the word feeds
// A-fragment register r of m16n8k16 for k-step kap of a 32-token block.
TQ_HD int vfield2(int kap, int r) { return ((kap ? 0x7463 : 0x5210) >> (4 * r)) & 0xF; }
TQ_HD int vfield4(int r) { return (0x3120 >> (4 * r)) & 0xF; }
// Effective mantissa position (after the decoder's shift) of the field for the low/high token half
// of a k-step; the decoder's B operand is prescaled by 2^(24 - pos).
TQ_HD constexpr int vpos2(int kap, int hiT) { return kap ? (hiT ? 8 : 6) : (hiT ? 4 : 0); }
TQ_HD constexpr int vpos4(int hiT) { return hiT ? 4 : 0; }

// Location of the value code of (token t, coordinate j) in VBITS: u32 word index and LSB of the field.
// A-fragment (m16n8k16, rows = coordinates, k = tokens) register r = rowhi + 2*hiT of lane (g, c)
// holds tokens (2c+8hiT, 2c+8hiT+1) in its two f16 halves e = token parity.
TQ_HD void vcode_loc(int d, int vb, int t, int j, int& word, int& bit) {
  const int blk = t >> 5, tau = t & 31, kap = tau >> 4, kk = tau & 15;
  const int c = (kk >> 1) & 3, e = kk & 1, hiT = kk >> 3;
  const int mt = j >> 4, g = j & 7, rowhi = (j >> 3) & 1;
  const int lane = 4 * g + c, r = rowhi + 2 * hiT;
  if (vb == 2) {
    word = (blk * (d >> 4) + mt) * 32 + lane;
    bit = 16 * e + 2 * vfield2(kap, r);
  } else {
    word = ((blk * (d >> 4) + mt) * 32 + lane) * 2 + kap;
    bit = 16 * e + 4 * vfield4(r);
  }
}

// Index (in fp16 units) of the value scale of (token t, group q) inside VSCALE.
TQ_HD int vscale_idx(int d, int t, int q) { return ((t >> 1) * (d / 32) + q) * 2 + (t & 1); }

// Byte offset of element (row n, column k) of a 128 x 128 bf16 matrix stored K-major in the
// tcgen05 canonical 128-byte-swizzled layout: two 64-column atoms of 128 rows; within an atom,
// 8-row groups of 1024 B, and the 16-byte chunk c of row r stored at chunk c ^ (r & 7).
// The same layout for a tile of `rows` rows (a multiple of 8): 64-column atoms of rows x 128 B.
TQ_HD uint32_t sw128_offset_rows(int n, int k, int rows) {
  return (uint32_t)((k >> 6) * rows * 128 + (n >> 3) * 1024 + (n & 7) * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) +
                    (k & 7) * 2);
}
TQ_HD uint32_t sw128_offset(int n, int k) {
  return (uint32_t)((k >> 6) * 16384 + (n >> 3) * 1024 + (n & 7) * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) +
                    (k & 7) * 2);
}

// Device tables (inside the caller's d_tables buffer). S_sw is S (rows = projection index,
// columns = coordinate) in the swizzled layout above; HD_sw is H diag(D) (entries +-1, bf16) in the
// same layout (head_dim 64 and 128: d rows, one or two 64-column atoms). For head_dim 256, S_sw holds S with 256 rows (sw128_offset_rows
// with 256 rows: four 32 KB atoms of 64 columns) and HD_sw holds H diag(D1) and H diag(D2) (128 x 128
// each) for the two halves of D, with H the 128-point Hadamard. S_frag is S in f16
// as m16n8k16 A fragments (see sfrag_idx), for the decode kernels' query projection.
struct TableOffsets {
  size_t D, S, St, cb, S_sw, HD_sw, S_frag, bytes;
};

// S_frag: [m-tile d/16][k-step d/16][lane 32] of {a0, a1, a2, a3} (four f16 pairs). Lane (g, c) of
// m-tile mt, k-step ks holds S[16mt + g (+8 for a1, a3)][16ks + 2c (+8 for a2, a3) + {0, 1}].
TQ_HD int sfrag_idx(int d, int mt, int ks, int lane) { return (mt * (d / 16) + ks) * 32 + lane; }
TableOffsets table_offsets(int d);

// Codebook block (floats). The index has kb - 1 bits, L = 2^(kb-1) levels.
//   cb[kCbCent ..]: the L centroids.
//   cb[kCbBnd ..]: the L - 1 boundaries.
//   cb[kCbW ..]: the weights of the +-1 index planes. The codebook is odd-symmetric, so
//     c[idx] = sum_p w_p (2 bit_p - 1), where the planes are:
//     - 2 bits: the high and low bit, with w = (c2 + c3)/2 and (c3 - c2)/2;
//     - 3 bits: b2, b1, b0 and b2^b1^b0, with w = A, B, C, E. These fit the upper levels c4..c7:
//       c = A + B t1 + C t0 + E t1 t0, where t = 2 bit - 1. The lower half follows by symmetry.
//   cb[kCbSmax]: max_i sum_j |S_ij| (rounded up).
constexpr int kCbCent = 0, kCbBnd = 8, kCbW = 16, kCbSmax = 20, kCbFloats = 32;

}  // namespace tq

struct tq_ctx {
  tq_config cfg;
  int device = -1;
  int sm_count = 0;
  bool host_only = false;
  tq::PageLayout pl;
  tq::TableOffsets to;
  int max_pages = 0;  // pages per (layer, slot, head)
  void* d_tables = nullptr;
  void* d_cache = nullptr;
  size_t cache_bytes = 0;
  size_t pages_off = 0, ring_off = 0, state_off = 0, acnt_off = 0, btab_off = 0, status_off = 0, total_bytes = 0;
  std::vector<float> D;
  std::vector<uint16_t> S;  // bf16 bits, row-major
  double cent[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // 2^(key_bits-1) used
  double bnd[7] = {0, 0, 0, 0, 0, 0, 0};
  // the last launch of this context, if it was a decode step: its layer (-1: none) and stream
  int step_layer = -1;
  void* step_stream = nullptr;
};

namespace tq {

// Pointers and sizes for one layer, passed to kernels by value.
struct LayerView {
  int d, vb, kb, G, Hkv, Hq, max_seqs, max_ctx, max_pages;
  uint32_t page_bytes;
  const float* D;
  const uint16_t* S;   // bf16 [d][d]
  const uint16_t* St;  // bf16 [d][d] transposed
  const float* cb;
  const uint16_t* S_sw;  // S in the tcgen05 swizzled K-major layout (head_dim 64, 128 and 256)
  const uint4* S_frag;   // S in f16 m16n8k16 A fragments (sfrag_idx)
  const uint16_t* HD_sw;  // H diag(D) (head_dim 64, 128; 256: H diag(D1), H diag(D2)) swizzled K-major
  uint8_t* pages;      // this layer: [slot][head][page][page_bytes], or paged: [block][head][page_bytes]
  const int32_t* btab; // paged cache: block table [slot][max_pages] (all layers); nullptr: contiguous
  int n_blocks;        // paged cache: blocks per layer
  uint16_t* ring;      // this layer: [slot][head][2][128][d] bf16
  int32_t* state;      // this layer: [slot][2] = {L, F}
  int32_t* acnt;       // this layer: [slot] arrival counters of the small-append kernel (left at zero)
  uint32_t* status;
};

LayerView layer_view(const tq_ctx* ctx, int layer);

// Decode workspace plan.
struct DecodePlan {
  int n_splits;        // history splits per (row, kv head); the ring is one extra split
  int pages_per_split;
  int wide;            // 1: the split CTAs run the wide variant (two page streams, two CTAs per SM)
  size_t part_off, part_stride;  // per (row, kv head, split) partial
  size_t cnt_off;                // per (row, kv head) int32 arrival counters at offset 0, room for
                                 // max_seqs rows (left at zero by every call)
  size_t row_cnt_off;            // per row int32 counters of the decode step's units (left at zero)
  size_t px_off;                 // tcgen05 prefill: expanded pages [row][KV head][px_pages][kPxBytes]
  int px_pages;                  // pages per (row, KV head) in that region
  size_t bytes;
};
// One page of one KV head expanded for the tcgen05 prefill: the f16 B tiles of the h, l and QJL planes
// (128 tokens x 128 coordinates) and V^T (128 coordinates x 128 tokens), 32 KB each in the tcgen05 128-byte
// swizzled K-major layout, then n_t as fp32 [128].
constexpr size_t kPxTileBytes = 32768, kPxBytes = 4 * kPxTileBytes + 512;
// cnt_rows: rows the arrival counters have room for (at least max_seqs; prefill rows per query).
DecodePlan decode_plan(const tq_ctx* ctx, int batch, int max_ctx_hint, int cnt_rows = 0, int ncol = kMaxG);

// Split-K decode CTAs resident per SM for ctx's (head_dim, value_bits), or for the wide variant (head_dim
// 128, K3/V2: two streams, two CTAs per SM); sets kernel attributes once.
int decode_resident_ctas(const tq_ctx* ctx, bool wide = false);
// Largest dynamic shared memory of one CTA on sm_103 (227 KB).
constexpr size_t kMaxSmemPerCta = 232448;
// True when the query-pair (prefill) decode kernel of ctx's shape fits kMaxSmemPerCta.
bool decode_pairs_fit(const tq_ctx* ctx);

// Records `msg` as the thread-local last error and returns `st` (for entry points outside tq_host.cpp).
tq_status set_error(tq_status st, const char* msg);
// True when ctx has a bound cache and `layer` is in range (sets the last error otherwise).
tq_status check_layer_ready(const tq_ctx* ctx, int layer);

cudaError_t launch_append(const tq_ctx* ctx, int layer, const void* k, const void* v, int dt,
                          const int32_t* seq_ids, const int32_t* n_new, int batch, int max_new, cudaStream_t s);
cudaError_t launch_flush(const tq_ctx* ctx, int layer, const int32_t* seq_ids, int batch, cudaStream_t s);
cudaError_t launch_reset(const tq_ctx* ctx, int layer, const int32_t* seq_ids, int batch, cudaStream_t s);
// phase -1 = the whole decode; 0 = zero the arrival counters, 1 = the decode launch. k_new / v_new
// (one token per row, dtype new_dt): a decode step that appends them in the same launch.
cudaError_t launch_decode(const tq_ctx* ctx, int layer, const void* q, float* out, const int32_t* seq_ids,
                          int batch, float scale, void* ws, const DecodePlan& plan, int phase, cudaStream_t s, int qpr = 1,
                          const int32_t* n_q = nullptr, int qp = 1, const void* k_new = nullptr,
                          const void* v_new = nullptr, int new_dt = 0, int late_state = 0);
// Prefill attention on tcgen05 (head_dim 128, key_bits 3, 4 query heads per KV head): the history
// partials of every (query, KV head), n_splits per unit, into the workspace in the decode's layout; then
// the exact ring split and the combine of every (query, KV head) into out.
bool prefill_tc_eligible(const tq_ctx* ctx);
int prefill_tc_splits(const tq_ctx* ctx, int batch, int q_per_row, int max_ctx_hint);
// Packed tokens [t0, t0 + count) of (layer, slot, KV head h) dequantised to fp32 k_hat, v_hat [count][d]
// (tq_dequantize_tokens).
cudaError_t launch_dequantize(const tq_ctx* ctx, int layer, int slot, int h, int t0, int count, int with_qjl,
                              float* k_out, float* v_out, cudaStream_t s);
cudaError_t launch_prefill_tc(const tq_ctx* ctx, int layer, const void* q, const int32_t* seq_ids, const int32_t* n_q,
                              int batch, int q_per_row, float scale, void* ws, const DecodePlan& plan, float* out,
                              cudaStream_t s);
// Decode launches read a row's state (and the pages it implies) before their stream wait. That is safe
// after every launch of this library except a decode step of the same layer on the same stream (it
// publishes the state at its end). step_follows() says whether the last launch of ctx on stream s was
// such a step (and forgets it); every launching entry point calls it, tq_decode_step then records itself.
bool step_follows(tq_ctx* ctx, int layer, cudaStream_t s);
void record_step(tq_ctx* ctx, int layer, cudaStream_t s);

}  // namespace tq
