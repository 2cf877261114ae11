// device_common.cuh -- small device helpers shared by the verification kernels:
// bulk-copy (TMA) + mbarrier wrappers, thread-block-cluster access, ordered
// keys for bf16/fp32 values, the exponent used for every softmax mass, and
// warp reductions.
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace specv {

namespace cg = cooperative_groups;

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes the barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// One-dimensional bulk copy global -> shared (the TMA engine), completing
// `bytes` of transaction count on `bar`.  dst, src and bytes must be
// multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Same, with the destination given as a shared-window address.
__device__ __forceinline__ void bulk_copy_g2s_addr(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Orders this thread's earlier shared-memory accesses before later writes by
// the async (bulk-copy) proxy to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Waits for phase `parity` of `bar` with a bounded number of polls.  Returns
// false if the limit was reached (the caller records a timeout status).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (it > 64) __nanosleep(64);
  }
  return false;
}

// Explicit shared-memory accesses through 32-bit shared-window addresses, so
// that the hot loops never fall back to generic addressing.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_u32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void sts_u16(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(static_cast<unsigned short>(v)) : "memory");
}
__device__ __forceinline__ void red_add_shared(uint32_t a, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
// Address of the same shared-memory location in cluster rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ double ld_cluster_f64(uint32_t a) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Streaming 16-byte global load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------------ element access

// Element traits: DT_BF16 rows hold 16-bit patterns, DT_F32 rows 32-bit floats.
template <int DT>
struct Elt;

template <>
struct Elt<DT_BF16> {
  static constexpr int kBytes = 2;
  static constexpr int kPerVec = 8;  // elements per 16-byte vector
  static constexpr int kKeyBits = 16;
  __device__ static __forceinline__ uint32_t bits_at(const void* base, int64_t i) {
    return static_cast<const uint16_t*>(base)[i];
  }
  // j-th element of a 16-byte vector
  __device__ static __forceinline__ uint32_t bits_of(const uint4& v, int j) {
    const uint32_t w = (j < 4) ? ((j < 2) ? v.x : v.y) : ((j < 6) ? v.z : v.w);
    return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
  }
  __device__ static __forceinline__ float value(uint32_t b) { return __uint_as_float(b << 16); }
  // Total-order key: larger value <=> larger key; -0 and +0 share one key.
  __device__ static __forceinline__ uint32_t key(uint32_t b) {
    if (b == 0x8000u) b = 0u;
    return (b & 0x8000u) ? (b ^ 0xFFFFu) : (b | 0x8000u);
  }
  __device__ static __forceinline__ uint32_t bits_of_key(uint32_t k) {
    return (k & 0x8000u) ? (k & 0x7FFFu) : (k ^ 0xFFFFu);
  }
  __device__ static __forceinline__ bool nonfinite_or_nan(uint32_t b) { return (b & 0x7F80u) == 0x7F80u; }
};

template <>
struct Elt<DT_F32> {
  static constexpr int kBytes = 4;
  static constexpr int kPerVec = 4;
  static constexpr int kKeyBits = 32;
  __device__ static __forceinline__ uint32_t bits_at(const void* base, int64_t i) {
    return static_cast<const uint32_t*>(base)[i];
  }
  __device__ static __forceinline__ uint32_t bits_of(const uint4& v, int j) {
    return (j < 2) ? ((j == 0) ? v.x : v.y) : ((j == 2) ? v.z : v.w);
  }
  __device__ static __forceinline__ float value(uint32_t b) { return __uint_as_float(b); }
  __device__ static __forceinline__ uint32_t key(uint32_t b) {
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  __device__ static __forceinline__ uint32_t bits_of_key(uint32_t k) {
    return (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  }
  __device__ static __forceinline__ bool nonfinite_or_nan(uint32_t b) {
    return (b & 0x7F800000u) == 0x7F800000u;
  }
};

// Softmax mass of a value relative to the row maximum:
//   exp((v - m) / T) = 2^((v - m) * log2(e) / T).
// Every mass in the sampling kernel (per element, per histogram bin, at the
// draft token) goes through this one function so that they agree bit for bit.
__device__ __forceinline__ float softmax_mass(float v, float m, float c_log2e_over_t) {
  return ex2_approx((v - m) * c_log2e_over_t);
}

// ------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ uint32_t warp_min_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = (w > v) ? w : v;
  }
  return v;
}

// Inclusive warp prefix sum (lane order).
__device__ __forceinline__ float warp_incl_scan(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float w = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += w;
  }
  return v;
}

__device__ __forceinline__ double warp_incl_scan_f64(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double w = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += w;
  }
  return v;
}

__device__ __forceinline__ uint32_t warp_incl_scan_u32(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t w = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += w;
  }
  return v;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  if (bits) atomicOr(status, bits);
}

}  // namespace specv
