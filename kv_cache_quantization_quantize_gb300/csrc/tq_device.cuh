// Device helpers shared by the libtq kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "tq_internal.h"

namespace tq {

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Coordinate that lane `lane` holds in x[e] when a d-vector is spread over one warp (NE = d / 32
// values per lane): 4 lane + e (+ 128 for e >= 4) for d >= 128, and 2 lane + e for d = 64.
template <int D>
__device__ __forceinline__ int lane_coord(int e, int lane) {
  return D == 64 ? 2 * lane + e : (e >> 2) * 128 + 4 * lane + (e & 3);
}

// Unnormalised Walsh-Hadamard transform (Sylvester order) of a d-vector spread over one warp in the
// lane_coord layout. The coordinate bits held in registers (bits 0-1 and, for d = 256, bit 7; bit 0
// for d = 64) are butterflied in registers, the lane bits across lanes with shuffles.
template <int NE>
__device__ __forceinline__ void warp_fwht(float (&x)[NE], int lane) {
#pragma unroll
  for (int base = 0; base + 3 < NE; base += 4) {
    float a0 = x[base + 0] + x[base + 1], a1 = x[base + 0] - x[base + 1];
    float a2 = x[base + 2] + x[base + 3], a3 = x[base + 2] - x[base + 3];
    x[base + 0] = a0 + a2;
    x[base + 2] = a0 - a2;
    x[base + 1] = a1 + a3;
    x[base + 3] = a1 - a3;
  }
  if (NE == 2) {  // head_dim 64: lane holds coordinates 2 lane + {0, 1}
    const float a = x[0], b = x[1];
    x[0] = a + b;
    x[1] = a - b;
  }
  if (NE == 8) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = x[e], b = x[4 + e];
      x[e] = a + b;
      x[4 + e] = a - b;
    }
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
      x[e] = upper ? (o - x[e]) : (x[e] + o);
    }
  }
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) { atomicOr(status, bit); }

// Address of packed page pg of (slot, KV head h) in layer view lv. A paged cache maps (slot, pg)
// through the block table; an entry outside [0, n_blocks) gives nullptr (the caller skips the page
// and reports TQ_DEV_ERR_BLOCK).
__device__ __forceinline__ uint8_t* page_addr(const LayerView& lv, int slot, int h, int pg) {
  if (!lv.btab) return lv.pages + (((size_t)slot * lv.Hkv + h) * lv.max_pages + pg) * lv.page_bytes;
  const int blk = lv.btab[(size_t)slot * lv.max_pages + pg];
  if (blk < 0 || blk >= lv.n_blocks) return nullptr;
  return lv.pages + ((size_t)blk * lv.Hkv + h) * lv.page_bytes;
}

// Barrier `id` (1..15) over the first `threads` threads that reach it (a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

// ---- mbarrier / bulk copy (async proxy) ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Shared -> global bulk copy (bytes a multiple of 16, both addresses 16-byte aligned) in the calling
// thread's bulk group; bulk_s2g_wait waits until every copy of the group has been written.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_s2g_wait() {
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}

// Plain arrival (no transaction bytes): completes a phase whose copy was not issued.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// Polls of a bounded mbarrier wait before it gives up (seconds of polling).
constexpr uint32_t kWaitPolls = 1u << 22;

// Bounded wait on an mbarrier phase: returns false after `limit` polls, never hangs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit = kWaitPolls) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Programmatic dependent launch. pdl_wait() blocks until the previous kernel in the stream has
// completed and its writes are visible (a no-op when launched without the PDL attribute).
// pdl_launch() lets the next kernel's CTAs be scheduled before this grid finishes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// Launches `kernel` with programmatic stream serialization allowed (see pdl_wait / pdl_launch).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace tq
