// Dequantisation of packed tokens back to the original basis (TurboQuant vLLM guide §二, steps 1-4, read
// backwards; §六 reports the fidelity of the result as a cosine similarity):
//   k_hat = n Pi^T (c[idx] + sqrt(pi/2)/d gamma S^T sigma)     (the QJL term optional)
//   v_hat = Pi^T ((code - 2^(b-1) + 1/2) s_g)
// with Pi^T = diag(D) H / sqrt(d), sigma = +-1 from the stored sign bits and (n, gamma, s_g) the stored fp16
// values. One warp per token, in the warp FWHT's coordinate layout (lane_coord); the page bits are read with
// the same location functions as the host's record conversion. Not on the decode path: it serves the
// fidelity report and tests.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kDqWarps = 8;  // tokens per CTA

template <int D>
__global__ void __launch_bounds__(32 * kDqWarps) k_dequantize(LayerView lv, int slot, int h, int t0, int count,
                                                              int with_qjl, float* k_out, float* v_out) {
  constexpr int NE = D / 32;  // coordinates per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int i = blockIdx.x * kDqWarps + warp;  // token of this warp, relative to t0
  if (i >= count) return;
  const int t = t0 + i, tt = t % kPage;
  const uint8_t* page = page_addr(lv, slot, h, t / kPage);
  float* ko = k_out + (size_t)i * D;
  float* vo = v_out + (size_t)i * D;
  if (!page) {  // a paged cache without a block for this page
    if (lane == 0) set_status(lv.status, TQ_DEV_ERR_BLOCK);
#pragma unroll
    for (int e = 0; e < NE; ++e) ko[lane_coord<D>(e, lane)] = vo[lane_coord<D>(e, lane)] = 0.f;
    return;
  }
  const PageLayout pl = page_layout(D, lv.vb, lv.kb);
  const uint32_t* kw = reinterpret_cast<const uint32_t*>(page + pl.kbits_off);
  const uint32_t* vw = reinterpret_cast<const uint32_t*>(page + pl.vbits_off);
  const uint16_t* vs = reinterpret_cast<const uint16_t*>(page + pl.vscale_off);
  const uint32_t nw = reinterpret_cast<const uint32_t*>(page + pl.norms_off)[tt];
  const float n = __half2float(__ushort_as_half((uint16_t)(nw & 0xffffu)));
  const float gamma = __half2float(__ushort_as_half((uint16_t)(nw >> 16)));
  const int mb = lv.kb - 1;  // index bits
  const float rs = rsqrtf((float)D);
  // ---- keys: y = c[idx] (+ kappa gamma S^T sigma), then n D (H y) / sqrt(d) ----
  float y[NE];
  uint32_t smask[NE];  // sign bits of coordinate lane_coord(e, l) in bit l
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    const int j = lane_coord<D>(e, lane);
    int idx = 0, w, b;
    for (int pi = 0; pi < mb; ++pi) {  // index bits, highest first
      kbit_loc(D, lv.kb, tt, j, pi, w, b);
      idx = 2 * idx + (int)((kw[w] >> b) & 1u);
    }
    kbit_loc(D, lv.kb, tt, j, mb, w, b);
    smask[e] = __ballot_sync(0xffffffffu, ((kw[w] >> b) & 1u) != 0u);
    y[e] = lv.cb[kCbCent + idx];
  }
  if (with_qjl) {
    // (S^T sigma)_j = sum_i sigma_i S[i][j]: coordinate i = lane_coord(e', l') has its sign at bit l' of smask[e']
    const float kappa = 1.2533141373155003f / (float)D;  // sqrt(pi/2) / d
    float acc[NE];
#pragma unroll
    for (int e = 0; e < NE; ++e) acc[e] = 0.f;
    for (int e2 = 0; e2 < NE; ++e2)
      for (int l2 = 0; l2 < 32; ++l2) {
        const int i2 = lane_coord<D>(e2, l2);
        const float sg = ((smask[e2] >> l2) & 1u) ? 1.f : -1.f;
        const uint16_t* row = lv.S + (size_t)i2 * D;
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[e] = fmaf(sg, bf16_to_f32(row[lane_coord<D>(e, lane)]), acc[e]);
      }
#pragma unroll
    for (int e = 0; e < NE; ++e) y[e] = fmaf(kappa * gamma, acc[e], y[e]);
  }
  warp_fwht<NE>(y, lane);
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    const int j = lane_coord<D>(e, lane);
    ko[j] = n * lv.D[j] * y[e] * rs;
  }
  // ---- values: x = (code - 2^(b-1) + 1/2) s_g, then D (H x) / sqrt(d) ----
  const int half = 1 << (lv.vb - 1);
  float x[NE];
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    const int j = lane_coord<D>(e, lane);
    int w, b;
    vcode_loc(D, lv.vb, tt, j, w, b);
    const int code = (int)((vw[w] >> b) & ((1u << lv.vb) - 1u));
    const float s = __half2float(__ushort_as_half(vs[vscale_idx(D, tt, j / 32)]));
    x[e] = ((float)(code - half) + 0.5f) * s;
  }
  warp_fwht<NE>(x, lane);
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    const int j = lane_coord<D>(e, lane);
    vo[j] = lv.D[j] * x[e] * rs;
  }
}

}  // namespace

cudaError_t launch_dequantize(const tq_ctx* ctx, int layer, int slot, int h, int t0, int count, int with_qjl,
                              float* k_out, float* v_out, cudaStream_t s) {
  if (count == 0) return cudaSuccess;
  const LayerView lv = layer_view(ctx, layer);
  const dim3 grid((count + kDqWarps - 1) / kDqWarps), block(32 * kDqWarps);
  switch (lv.d) {
    case 64:
      k_dequantize<64><<<grid, block, 0, s>>>(lv, slot, h, t0, count, with_qjl, k_out, v_out);
      break;
    case 128:
      k_dequantize<128><<<grid, block, 0, s>>>(lv, slot, h, t0, count, with_qjl, k_out, v_out);
      break;
    default:
      k_dequantize<256><<<grid, block, 0, s>>>(lv, slot, h, t0, count, with_qjl, k_out, v_out);
      break;
  }
  return cudaGetLastError();
}

}  // namespace tq
