// Quantize-on-append ([Guide] §二, five-step pipeline): one CTA writes one packed page (128 tokens of
// one KV head). This is the CUDA-core path for ring flushes and appends. The QJL projection z = S r
// is an fp32 FMA contraction against S^T staged in shared memory.
#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kQThreads = 256;  // 8 warps; warp w quantises tokens w, w + 8, ...

struct AppendArgs {
  LayerView lv;
  const void* k;
  const void* v;
  int dt;  // 0 = bf16, 1 = f32
  const int32_t* seq_ids;
  const int32_t* n_new;
  int max_new;
  int flush;  // 1: quantise the current ring block (tq_ring_flush)
};

// Load 4 consecutive coordinates of one token of the source stream (ring bf16 or input bf16/f32).
__device__ __forceinline__ void load4(const AppendArgs& a, int which, int slot, int b, int h, int pos, int L, int Np,
                                      int j, float (&o)[4]) {
  const int d = a.lv.d;
  if (pos < L) {  // still in the ring: ring index pos - Np
    const uint16_t* src = a.lv.ring + ((((size_t)slot * a.lv.Hkv + h) * 2 + which) * kPage + (pos - Np)) * d + j;
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    o[0] = __uint_as_float(u.x << 16);
    o[1] = __uint_as_float(u.x & 0xffff0000u);
    o[2] = __uint_as_float(u.y << 16);
    o[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    const size_t off = (((size_t)b * a.max_new + (pos - L)) * a.lv.Hkv + h) * d + j;
    const void* base = which ? a.v : a.k;
    if (a.dt == 0) {
      const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + off);
      o[0] = __uint_as_float(u.x << 16);
      o[1] = __uint_as_float(u.x & 0xffff0000u);
      o[2] = __uint_as_float(u.y << 16);
      o[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
      const float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
      o[0] = f.x;
      o[1] = f.y;
      o[2] = f.z;
      o[3] = f.w;
    }
  }
}

// Which page this CTA writes, from the sequence state. Returns false when the CTA has no work.
__device__ __forceinline__ bool page_task(const AppendArgs& a, int b, int j, int& slot, int& L, int& Np, int& pg,
                                          int& valid, bool report) {
  slot = a.seq_ids[b];
  if (slot < 0 || slot >= a.lv.max_seqs) {
    if (report) set_status(a.lv.status, TQ_DEV_ERR_SEQ_ID);
    return false;
  }
  L = a.lv.state[2 * slot];
  Np = L > 0 ? kPage * ((L - 1) / kPage) : 0;
  if (a.flush) {
    const int R = L - Np;
    if (R <= 0 || j > 0) return false;
    pg = Np / kPage;
    valid = R;
    return true;
  }
  const int nn = a.n_new[b];
  const int L2 = L + nn;
  if (nn < 0 || nn > a.max_new || L2 > a.lv.max_ctx) {
    if (report) set_status(a.lv.status, TQ_DEV_ERR_CAPACITY);
    return false;
  }
  const int Np2 = L2 > 0 ? kPage * ((L2 - 1) / kPage) : 0;
  if (j >= (Np2 - Np) / kPage) return false;
  pg = Np / kPage + j;
  valid = kPage;
  return true;
}

template <int D>
__global__ void __launch_bounds__(kQThreads) k_quantize_pages(AppendArgs a) {
  constexpr int NE = D / 32;  // coordinates per lane
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* st2 = reinterpret_cast<uint32_t*>(smem);                    // S^T as bf16 pairs [D][D/2]
  uint8_t* kcode = smem + 2 * D * D;                                    // [128][D]: idx | sign << 2
  uint8_t* vcode = kcode + kPage * D;                                   // [128][D]
  uint32_t* norms = reinterpret_cast<uint32_t*>(vcode + kPage * D);     // [128] n16 | gamma16 << 16
  uint16_t* scales = reinterpret_cast<uint16_t*>(norms + kPage);        // [128][D/32]
  float* rbuf = reinterpret_cast<float*>(scales + kPage * (D / 32));    // [8 warps][D]

  const int b = blockIdx.x, h = blockIdx.y;
  pdl_wait();  // sequence state, ring and inputs come from earlier work on the stream
  pdl_launch();
  int slot, L, Np, pg, valid;
  if (!page_task(a, b, blockIdx.z, slot, L, Np, pg, valid, h == 0 && blockIdx.z == 0 && threadIdx.x == 0)) return;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const LayerView& lv = a.lv;
  // stage S^T (bf16) in shared memory
  {
    const uint4* src = reinterpret_cast<const uint4*>(lv.St);
    uint4* dst = reinterpret_cast<uint4*>(st2);
    for (int i = tid; i < D * D / 8; i += kQThreads) dst[i] = src[i];
  }
  float Dv[NE], cent[4], bnd[3];
#pragma unroll
  for (int e = 0; e < NE; ++e) Dv[e] = lv.D[(e >> 2) * 128 + 4 * lane + (e & 3)];
#pragma unroll
  for (int i = 0; i < 4; ++i) cent[i] = lv.cb[i];
#pragma unroll
  for (int i = 0; i < 3; ++i) bnd[i] = lv.cb[4 + i];
  __syncthreads();

  const int vb = lv.vb, vhalf = 1 << (vb - 1);
  const float inv_sqrt_d = rsqrtf((float)D);
  float* r = rbuf + warp * D;
  for (int t = warp; t < kPage; t += kQThreads / 32) {
    const int pos = pg * kPage + t;
    float x[NE], y[NE];
    if (t < valid) {
#pragma unroll
      for (int hh = 0; hh < NE / 4; ++hh) {
        float o[4];
        load4(a, 0, slot, b, h, pos, L, Np, 128 * hh + 4 * lane, o);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[4 * hh + e] = o[e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < NE; ++e) x[e] = 0.f;
    }
    // ---- key: n = ||k||, y = Pi k / n, Lloyd-Max index, residual, gamma ----
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < NE; ++e) ss = fmaf(x[e], x[e], ss);
    ss = warp_sum(ss);
    const float n = sqrtf(ss);
#pragma unroll
    for (int e = 0; e < NE; ++e) y[e] = x[e] * Dv[e];
    warp_fwht<NE>(y, lane);
    const float scale = n > 0.f ? 1.0f / (n * sqrtf((float)D)) : 0.f;
    float rr = 0.f;
    uint8_t* kc = kcode + t * D;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const float yy = y[e] * scale;
      const int idx = (yy > bnd[0]) + (yy > bnd[1]) + (yy > bnd[2]);
      const float res = yy - cent[idx];
      rr = fmaf(res, res, rr);
      const int j = (e >> 2) * 128 + 4 * lane + (e & 3);
      r[j] = res;
      kc[j] = (uint8_t)idx;
    }
    rr = warp_sum(rr);
    const float gamma = sqrtf(rr);
    __syncwarp();
    // ---- QJL: z = S r; lane owns rows 2l, 2l+1 (+64m) ----
    {
      constexpr int NR = D / 64;  // row pairs per lane
      float z0[NR], z1[NR];
#pragma unroll
      for (int m = 0; m < NR; ++m) z0[m] = z1[m] = 0.f;
      for (int jj = 0; jj < D; ++jj) {
        const float rj = r[jj];
#pragma unroll
        for (int m = 0; m < NR; ++m) {
          const uint32_t s = st2[jj * (D / 2) + lane + 32 * m];
          z0[m] = fmaf(__uint_as_float(s << 16), rj, z0[m]);
          z1[m] = fmaf(__uint_as_float(s & 0xffff0000u), rj, z1[m]);
        }
      }
      __syncwarp();
#pragma unroll
      for (int m = 0; m < NR; ++m) {
        const int i0 = 2 * lane + 64 * m;
        kc[i0] = (uint8_t)(kc[i0] | ((z0[m] >= 0.f) << 2));
        kc[i0 + 1] = (uint8_t)(kc[i0 + 1] | ((z1[m] >= 0.f) << 2));
      }
    }
    if (lane == 0) {
      const __half nh = __float2half_rn(fminf(n, 65504.f)), gh = __float2half_rn(gamma);
      norms[t] = (uint32_t)__half_as_ushort(nh) | ((uint32_t)__half_as_ushort(gh) << 16);
    }
    // ---- value: v' = Pi v, symmetric mid-rise groups of 32, fp16 scale ----
    if (t < valid) {
#pragma unroll
      for (int hh = 0; hh < NE / 4; ++hh) {
        float o[4];
        load4(a, 1, slot, b, h, pos, L, Np, 128 * hh + 4 * lane, o);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[4 * hh + e] = o[e] * Dv[4 * hh + e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < NE; ++e) x[e] = 0.f;
    }
    warp_fwht<NE>(x, lane);
    uint8_t* vc = vcode + t * D;
#pragma unroll
    for (int hh = 0; hh < NE / 4; ++hh) {
      float am = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[4 * hh + e] *= inv_sqrt_d;
        am = fmaxf(am, fabsf(x[4 * hh + e]));
      }
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
      const float s32 = fminf(__fdiv_rn(am, (float)vhalf - 0.5f), 65504.f);
      const __half sh = __float2half_rn(s32);
      const float s = __half2float(sh);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int code = vhalf;
        if (s > 0.f) {
          const float qv = floorf(__fdiv_rn(x[4 * hh + e], s));
          code = (int)fminf(fmaxf(qv, (float)-vhalf), (float)(vhalf - 1)) + vhalf;
        }
        vc[128 * hh + 4 * lane + e] = (uint8_t)code;
      }
      if ((lane & 7) == 0) scales[t * (D / 32) + 4 * hh + (lane >> 3)] = __half_as_ushort(sh);
    }
  }
  __syncthreads();

  // ---- pack the page (fragment-major layout) ----
  uint8_t* page = lv.pages + (((size_t)slot * lv.Hkv + h) * lv.max_pages + pg) * lv.page_bytes;
  const PageLayout pl = page_layout(D, vb);
  uint32_t* kw = reinterpret_cast<uint32_t*>(page + pl.kbits_off);
  constexpr int HALVES = D / 128;
  for (int w = tid; w < 8 * 3 * HALVES * 32 * 2; w += kQThreads) {
    const int r = w & 1, ln = (w >> 1) & 31, hf = (w >> 6) % HALVES, pi = (w / (64 * HALVES)) % 3;
    const int tile = w / (192 * HALVES);
    const int t = 16 * tile + (ln >> 2) + 8 * r, c = ln & 3;
    const uint8_t* kc = kcode + t * D + 128 * hf + 2 * c;
    uint32_t word = 0;
#pragma unroll
    for (int sq = 0; sq < 8; ++sq)
#pragma unroll
      for (int sub = 0; sub < 2; ++sub)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int code = kc[16 * sq + 8 * sub + e];
          const int bit = pi == 0 ? (code >> 1) & 1 : pi == 1 ? code & 1 : (code >> 2) & 1;
          word |= (uint32_t)bit << (2 * sq + sub + 16 * e);
        }
    kw[w] = word;
  }
  uint32_t* nw = reinterpret_cast<uint32_t*>(page + pl.norms_off);
  for (int t = tid; t < kPage; t += kQThreads) nw[t] = norms[t];
  uint32_t* vw = reinterpret_cast<uint32_t*>(page + pl.vbits_off);
  if (vb == 2) {
    for (int w = tid; w < 4 * (D / 16) * 32; w += kQThreads) {
      const int ln = w & 31, mt = (w >> 5) % (D / 16), blk = w / (32 * (D / 16));
      const int g = ln >> 2, c = ln & 3;
      uint32_t word = 0;
#pragma unroll
      for (int kap = 0; kap < 2; ++kap)
#pragma unroll
        for (int rg = 0; rg < 4; ++rg)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int t = 32 * blk + 16 * kap + 8 * (rg >> 1) + 2 * c + e;
            const int j = 16 * mt + 8 * (rg & 1) + g;
            word |= (uint32_t)vcode[t * D + j] << (16 * e + 2 * vfield2(kap, rg));
          }
      vw[w] = word;
    }
  } else {
    for (int w = tid; w < 4 * (D / 16) * 32 * 2; w += kQThreads) {
      const int kap = w & 1, ln = (w >> 1) & 31, mt = (w >> 6) % (D / 16), blk = w / (64 * (D / 16));
      const int g = ln >> 2, c = ln & 3;
      uint32_t word = 0;
#pragma unroll
      for (int rg = 0; rg < 4; ++rg)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 32 * blk + 16 * kap + 8 * (rg >> 1) + 2 * c + e;
          const int j = 16 * mt + 8 * (rg & 1) + g;
          word |= (uint32_t)vcode[t * D + j] << (16 * e + 4 * vfield4(rg));
        }
      vw[w] = word;
    }
  }
  uint16_t* sw = reinterpret_cast<uint16_t*>(page + pl.vscale_off);
  for (int i = tid; i < kPage * (D / 32); i += kQThreads) sw[vscale_idx(D, i / (D / 32), i % (D / 32))] = scales[i];
}

// Ring update after the quantise launch: write the new ring tail and the sequence state.
__global__ void __launch_bounds__(256) k_ring_update(AppendArgs a) {
  const int b = blockIdx.x;
  pdl_wait();  // the quantise launch has read the old ring and state
  pdl_launch();
  const LayerView& lv = a.lv;
  const int slot = a.seq_ids[b];
  if (slot < 0 || slot >= lv.max_seqs) return;
  const int L = lv.state[2 * slot], F = lv.state[2 * slot + 1];
  const int Np = L > 0 ? kPage * ((L - 1) / kPage) : 0;
  if (a.flush) {
    __syncthreads();
    if (threadIdx.x == 0) lv.state[2 * slot + 1] = L - Np;
    return;
  }
  const int nn = a.n_new[b];
  const int L2 = L + nn;
  if (nn < 0 || nn > a.max_new || L2 > lv.max_ctx) return;
  const int Np2 = L2 > 0 ? kPage * ((L2 - 1) / kPage) : 0;
  const int p0 = max(L, Np2);
  const int d = lv.d, q4 = d / 4;
  const int n_items = (L2 - p0) * lv.Hkv * 2 * q4;  // (pos, head, which, quad)
  for (int it = threadIdx.x; it < n_items; it += blockDim.x) {
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
  __syncthreads();
  if (threadIdx.x == 0) {
    lv.state[2 * slot] = L2;
    lv.state[2 * slot + 1] = Np2 > Np ? 0 : F;
  }
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
  return 2 * D * D + 2 * kPage * D + 4 * kPage + 2 * kPage * (D / 32) + 4 * 8 * D;
}

template <int D>
cudaError_t launch_quantize_d(const AppendArgs& a, int batch, int pages, cudaStream_t s) {
  const size_t smem = quantize_smem_bytes<D>();
  static bool attr_set = false;  // set once, outside any stream capture that follows
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_quantize_pages<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(batch, a.lv.Hkv, pages);
  return launch_pdl(k_quantize_pages<D>, grid, dim3(kQThreads), smem, s, a);
}

cudaError_t launch_quantize(const AppendArgs& a, int batch, int pages, cudaStream_t s) {
  if (a.lv.d == 128) return launch_quantize_d<128>(a, batch, pages, s);
  return launch_quantize_d<256>(a, batch, pages, s);
}

}  // namespace

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
  const int pages = (max_new + kPage - 1) / kPage;
  cudaError_t e = launch_quantize(a, batch, pages, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_ring_update, dim3(batch), dim3(256), 0, s, a);
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
