// sample_kernel.cu -- speculative-sampling verification on sm_103a.
//
// What it computes (Edge Inference Notes, post on speculative decoding and
// EAGLE-3, "The core idea: draft, then check", step 3, and "Why it changes
// nothing about the output"): for every sequence b and draft position i,
// p_i and q_i are the temperature-scaled, top-k / top-p filtered softmax of
// the target and draft rows; draft x_i is accepted iff u_i * q_i(x_i) <
// p_i(x_i); at the first rejection n one token is drawn from
// max(0, p_n - q_n) with u_{k+1}, else a bonus token from p_k with u_k.
//
// How (one GPU, memory-bound).  One CTA owns one unit (b, i) and streams its
// target row and draft row from HBM exactly once, 16-byte loads by warp
// segments in index order.  While streaming, for each row:
//   - masses are taken on a power-of-two lattice: with c = log2(e) / T and
//     an integer k_t >= max(l) * c held per thread, mass(l) = 2^(l c - k_t)
//     (one packed f32x2 fma and one ex2 per element).  Raising k_t rescales
//     the running sum by an exact power of two, so the row sum
//     Z = sum 2^(l c - K) (K the CTA-wide k) carries no rescaling error;
//     2^(l c - K) / Z is the softmax of l / T.
//   - every element within kTheta octaves of mass of the running maximum is
//     appended to its warp's candidate list (index order; entries below the
//     current bound are purged when a list fills).  A top-k / top-p cut
//     within kTheta octaves of the maximum is therefore decided from the
//     lists alone: a histogram of exact values, a four-warp scan for the cut,
//     its tie count and the kept normaliser.  Rows whose cut lies deeper
//     (flat rows), fp32 rows and overflowing lists take an exact bitwise
//     search over the keys that re-reads the row.
// The accept test reads p(x_i), q(x_i) at x_i.  The residual max(0, p - q)
// (or the bonus p) is non-zero only on the kept set of p, which the lists
// hold in index order: per-warp sums, a prefix over warps and a walk of one
// list give the drawn token.  Every unit draws (the residual draw is
// speculative), so no row is read twice on the fast path.  The last writer
// of a sequence (atomic ticket, no spin-wait) applies the first-rejection
// rule and commits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "device_common.cuh"

namespace specv {

__device__ void sample_finalize(const SampleArgs& a, int b);

namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
using u64 = unsigned long long;

constexpr int kListCap = 800;                       // candidate entries per warp per row
constexpr int kSyncEvery = 4;                       // stream iterations between CTA maximum exchanges
constexpr float kTheta = 13.f;                      // octaves of mass kept as candidates
constexpr uint32_t kSlotMask = static_cast<uint32_t>(kWindow) - 1u;
constexpr int kGroups = kWindow / 4;                // aligned groups of four keys
constexpr int kScanWarps = 4;                       // warps that scan one row's histogram
constexpr int kSegBits = 16;                        // element index within a warp segment

// ------------------------------------------------------- packed f32x2 math

__device__ __forceinline__ u64 pk2(uint32_t x, uint32_t y) {
  u64 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(x), "r"(y));
  return r;
}
__device__ __forceinline__ u64 pkf(float x, float y) { return pk2(__float_as_uint(x), __float_as_uint(y)); }
__device__ __forceinline__ void upk(u64 r, float& x, float& y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(r));
}
__device__ __forceinline__ u64 add2(u64 a, u64 b) {
  u64 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
  u64 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// 2^(l c - k) for both halves: the lattice masses of two elements
__device__ __forceinline__ u64 lat2(u64 l2, u64 c2, u64 nk2) {
  float x, y;
  upk(fma2(l2, c2, nk2), x, y);
  return pkf(ex2_approx(x), ex2_approx(y));
}
// The lattice mass of one value: every mass of the kernel goes through this
// function or lat2 (same fma, same ex2), so they agree bit for bit.
__device__ __forceinline__ float lat_mass(float l, float c, float k) { return ex2_approx(fmaf(l, c, -k)); }

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ int warp_max_i32(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// 2^d for an integer d, exact (0 below the normal range).
__device__ __forceinline__ float exp2i(int d) {
  return d < -126 ? 0.f : __int_as_float((127 + min(d, 127)) << 23);
}

// Double-float: an unevaluated sum hi + lo of two floats (about 48 bits),
// kept with fp32 instructions only (the fp64 pipe of this GPU is narrow).
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF df_from(double d) {
  const float h = static_cast<float>(d);
  return DF{h, static_cast<float>(d - static_cast<double>(h))};
}
// a + b by the error-free two-sum of the high parts
__device__ __forceinline__ DF df_add(DF a, float b) {
  const float s = a.hi + b;
  const float bb = s - a.hi;
  const float e = ((a.hi - (s - bb)) + (b - bb)) + a.lo;
  const float h = s + e;
  return DF{h, e - (h - s)};
}
__device__ __forceinline__ DF df_add2(DF a, DF b) { return df_add(df_add(a, b.hi), b.lo); }
__device__ __forceinline__ DF df_neg(DF a) { return DF{-a.hi, -a.lo}; }
__device__ __forceinline__ DF df_shfl_up(DF a, int o) {
  return DF{__shfl_up_sync(kFull, a.hi, o), __shfl_up_sync(kFull, a.lo, o)};
}
__device__ __forceinline__ DF df_shfl(DF a, int l) { return DF{__shfl_sync(kFull, a.hi, l), __shfl_sync(kFull, a.lo, l)}; }
__device__ __forceinline__ DF warp_incl_scan_df(DF v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF w = df_shfl_up(v, o);
    if (lane >= o) v = df_add2(v, w);
  }
  return v;
}
// a * b for a double-float and a float
__device__ __forceinline__ DF df_mul_f(DF a, float b) {
  const float p = a.hi * b;
  const float e = fmaf(a.hi, b, -p) + a.lo * b;
  const float h = p + e;
  return DF{h, e - (h - p)};
}
__device__ __forceinline__ bool df_lt(DF a, DF b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }
__device__ __forceinline__ float df_float(DF a) { return a.hi + a.lo; }
__device__ __forceinline__ double df_double(DF a) { return static_cast<double>(a.hi) + static_cast<double>(a.lo); }

// ------------------------------------------------- per-dtype vector kernels

template <int DT>
struct Hot;

template <>
struct Hot<DT_BF16> {
  __device__ static __forceinline__ __nv_bfloat162 b2(uint32_t w) {
    __nv_bfloat162 r;
    *reinterpret_cast<uint32_t*>(&r) = w;
    return r;
  }
  static constexpr uint32_t kPad = 0xFF80FF80u;  // -inf, -inf
  __device__ static __forceinline__ float vmax(const uint4& v) {
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(b2(v.x), b2(v.y)), __hmax2_nan(b2(v.z), b2(v.w)));
    return max_nan(__low2float(m), __high2float(m));
  }
  __device__ static __forceinline__ void mass_vec(const uint4& v, u64 c2, u64 nk2, u64& acc0, u64& acc1) {
    acc0 = add2(acc0, lat2(pk2(v.x << 16, v.x & 0xFFFF0000u), c2, nk2));
    acc1 = add2(acc1, lat2(pk2(v.y << 16, v.y & 0xFFFF0000u), c2, nk2));
    acc0 = add2(acc0, lat2(pk2(v.z << 16, v.z & 0xFFFF0000u), c2, nk2));
    acc1 = add2(acc1, lat2(pk2(v.w << 16, v.w & 0xFFFF0000u), c2, nk2));
  }
  __device__ static __forceinline__ uint32_t thr_pack(uint32_t bits) { return bits | (bits << 16); }
  __device__ static __forceinline__ uint32_t mask_ge(const uint4& v, uint32_t thr) {
    const __nv_bfloat162 t = b2(thr);
    const uint32_t m0 = __hge2_mask(b2(v.x), t), m1 = __hge2_mask(b2(v.y), t);
    const uint32_t m2 = __hge2_mask(b2(v.z), t), m3 = __hge2_mask(b2(v.w), t);
    return (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) | ((m2 & 1u) << 4) |
           ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u);
  }
  __device__ static __forceinline__ uint32_t mask_eq(const uint4& v, uint32_t thr) {
    const __nv_bfloat162 t = b2(thr);
    const uint32_t m0 = __heq2_mask(b2(v.x), t), m1 = __heq2_mask(b2(v.y), t);
    const uint32_t m2 = __heq2_mask(b2(v.z), t), m3 = __heq2_mask(b2(v.w), t);
    return (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) | ((m2 & 1u) << 4) |
           ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u);
  }
};

template <>
struct Hot<DT_F32> {
  static constexpr uint32_t kPad = 0xFF800000u;
  __device__ static __forceinline__ float vmax(const uint4& v) {
    return max_nan(max_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                   max_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
  __device__ static __forceinline__ void mass_vec(const uint4& v, u64 c2, u64 nk2, u64& acc0, u64& acc1) {
    acc0 = add2(acc0, lat2(pk2(v.x, v.y), c2, nk2));
    acc1 = add2(acc1, lat2(pk2(v.z, v.w), c2, nk2));
  }
  __device__ static __forceinline__ uint32_t thr_pack(uint32_t bits) { return bits; }
  __device__ static __forceinline__ uint32_t mask_ge(const uint4& v, uint32_t thr) {
    const float t = __uint_as_float(thr);
    return (__uint_as_float(v.x) >= t ? 1u : 0u) | (__uint_as_float(v.y) >= t ? 2u : 0u) |
           (__uint_as_float(v.z) >= t ? 4u : 0u) | (__uint_as_float(v.w) >= t ? 8u : 0u);
  }
  __device__ static __forceinline__ uint32_t mask_eq(const uint4& v, uint32_t thr) {
    const float t = __uint_as_float(thr);
    return (__uint_as_float(v.x) == t ? 1u : 0u) | (__uint_as_float(v.y) == t ? 2u : 0u) |
           (__uint_as_float(v.z) == t ? 4u : 0u) | (__uint_as_float(v.w) == t ? 8u : 0u);
  }
};

// ------------------------------------------------------------ row state

template <int DT>
__device__ __forceinline__ float value_of_key(uint32_t k) {
  return Elt<DT>::value(Elt<DT>::bits_of_key(k));
}
template <int DT>
__device__ __forceinline__ uint32_t key_of_float(float v) {
  const uint32_t b = (Elt<DT>::kBytes == 2) ? (__float_as_uint(v) >> 16) : __float_as_uint(v);
  return Elt<DT>::key(b);
}
// Smallest bf16 / fp32 value not below v (v finite), as bits.
template <int DT>
__device__ __forceinline__ uint32_t bits_round_up(float v) {
  const uint32_t u = __float_as_uint(v);
  if (DT == DT_F32) return u;
  const uint32_t hi = u >> 16;
  if ((u & 0xFFFFu) == 0u) return hi;
  return (u & 0x80000000u) ? hi : hi + 1u;  // negative: toward zero is up
}
// Largest bf16 / fp32 value not above v, as bits.
template <int DT>
__device__ __forceinline__ uint32_t bits_round_down(float v) {
  const uint32_t u = __float_as_uint(v);
  if (DT == DT_F32) return u;
  const uint32_t hi = u >> 16;
  if ((u & 0xFFFFu) == 0u) return hi;
  return (u & 0x80000000u) ? hi + 1u : hi;  // negative: away from zero is down
}

// The kept set of a row: key > kstar, or key == kstar and index < tie_cut.
struct RowStat {
  float c;               // log2(e) / T
  float K;               // lattice exponent (integer) of the row: masses 2^(l c - K)
  float m;               // row maximum
  uint32_t kmax;         // key of m
  uint32_t kstar;
  int tie_cut;           // row index bound for tokens of value kstar
  float inv_z;           // 1 / mass of the kept set
  float zkept;
  int all_kept;
  int covered;           // the candidate lists hold every kept token
  int bad;
};

__device__ __forceinline__ bool kept_key(const RowStat& rs, uint32_t key, int j) {
  if (rs.all_kept) return true;
  if (key > rs.kstar) return true;
  return key == rs.kstar && j < rs.tie_cut;
}

template <int DT>
__device__ __forceinline__ float prob_of(const RowStat& rs, uint32_t bits, int j) {
  using E = Elt<DT>;
  return kept_key(rs, E::key(bits), j) ? lat_mass(E::value(bits), rs.c, rs.K) * rs.inv_z : 0.f;
}

struct CutOut {
  uint32_t kstar;        // key of the last kept value
  uint32_t keep;         // tokens of value kstar that are kept (lowest indices)
  uint32_t total;        // tokens of value kstar in the row
  int found;
  DF zkept;              // mass of the kept set
};

struct Shm {
  float w_m[kWarps][2];
  int w_k[kWarps][2];
  float w_z[kWarps][2];
  uint32_t w_n[kWarps][2];     // candidate list lengths
  uint32_t w_floor[kWarps][2]; // key above which a warp's list is complete
  float x_m[2][kWarps][2];     // running maxima exchanged while streaming (double-buffered)
  float w_s[kWarps];
  float w_sp[kWarps];
  uint32_t w_u[kWarps][2];
  double w_d[kWarps];
  uint32_t s_C[2][kScanWarps];
  DF s_M[2][kScanWarps];
  DF z[2];                     // row sums of masses
  CutOut cutk[2];
  CutOut cut[2];
  uint32_t klo[2];
  int tie_warp[2];
  uint32_t tie_j[2];
  int tie_cut[2];
  RowStat rs[2];
  int draw_warp;
  float draw_base;
  double red_d;
  uint32_t red_u, red_k;
};

// 16-byte vector v of a row (elements v*kPerVec ...), -inf beyond n.
template <int DT>
__device__ __forceinline__ uint4 load_vec(const unsigned char* row, int v, int n, bool aligned) {
  using E = Elt<DT>;
  if (aligned && (v + 1) * E::kPerVec <= n) return ldg_stream(row + 16 * static_cast<size_t>(v));
  uint32_t w[4] = {Hot<DT>::kPad, Hot<DT>::kPad, Hot<DT>::kPad, Hot<DT>::kPad};
#pragma unroll
  for (int j = 0; j < E::kPerVec; ++j) {
    const int t = v * E::kPerVec + j;
    if (t < n) {
      const uint32_t b = E::bits_at(row, t);
      if (E::kBytes == 2) {
        const int q = j >> 1;
        w[q] = (j & 1) ? ((w[q] & 0xFFFFu) | (b << 16)) : ((w[q] & 0xFFFF0000u) | b);
      } else {
        w[j] = b;
      }
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Bit j set for the elements of vector v that lie inside a row of n.
template <int DT>
__device__ __forceinline__ uint32_t vmask(int v, int n) {
  const int left = n - v * Elt<DT>::kPerVec;
  return left >= Elt<DT>::kPerVec ? (1u << Elt<DT>::kPerVec) - 1u : (left > 0 ? (1u << left) - 1u : 0u);
}

// ------------------------------------------------------ CTA reductions

// Fixed-order CTA sums (deterministic); every thread gets the result.
__device__ __forceinline__ DF block_sum_df(float v, Shm& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_f32(v);
  if (lane == 0) sh.w_s[warp] = v;
  __syncthreads();
  DF t{0.f, 0.f};
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t = df_add(t, sh.w_s[w]);
  __syncthreads();
  return t;
}
__device__ __forceinline__ uint32_t block_sum_u32(uint32_t v, Shm& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_u32(v);
  if (lane == 0) sh.w_u[warp][0] = v;
  __syncthreads();
  uint32_t t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += sh.w_u[w][0];
  __syncthreads();
  return t;
}
__device__ __forceinline__ uint32_t block_min_u32(uint32_t v, Shm& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_min_u32(v);
  if (lane == 0) sh.w_u[warp][1] = v;
  __syncthreads();
  uint32_t t = 0xFFFFFFFFu;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t = min(t, sh.w_u[w][1]);
  __syncthreads();
  return t;
}

// ------------------------------------------------- exact search by passes

enum PassKind { PASS_COUNT_GE = 0, PASS_MASS_GT = 1, PASS_MIN_GE = 2, PASS_COUNT_EQ = 3 };

// One pass over a whole row (re-read from global memory), reduced over the
// CTA.  Used by rows whose cut is not decided from the candidate lists.
template <int DT>
__device__ __noinline__ double row_pass(Shm& sh, const unsigned char* row, int V, bool aligned, int kind,
                                        uint32_t kappa, const RowStat& rs) {
  using E = Elt<DT>;
  const int nvec = (V + E::kPerVec - 1) / E::kPerVec;
  uint32_t cnt = 0, kmin = 0xFFFFFFFFu;
  float mass = 0.f;
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    const uint4 x = load_vec<DT>(row, v, V, aligned);
#pragma unroll
    for (int j = 0; j < E::kPerVec; ++j) {
      if (v * E::kPerVec + j < V) {
        const uint32_t b = E::bits_of(x, j);
        const uint32_t k = E::key(b);
        if (kind == PASS_COUNT_GE) cnt += (k >= kappa);
        else if (kind == PASS_COUNT_EQ) cnt += (k == kappa);
        else if (kind == PASS_MIN_GE) { if (k >= kappa) kmin = min(kmin, k); }
        else if (k > kappa) mass += lat_mass(E::value(b), rs.c, rs.K);
      }
    }
  }
  if (kind == PASS_MASS_GT) return df_double(block_sum_df(mass, sh));
  if (kind == PASS_MIN_GE) return static_cast<double>(block_min_u32(kmin, sh));
  return static_cast<double>(block_sum_u32(cnt, sh));
}

// The exact cut of one row by a bitwise search over the keys.
template <int DT>
__device__ __noinline__ CutOut search_cut(Shm& sh, const unsigned char* row, int V, bool aligned, int top_k,
                                          float top_p, const RowStat& rs, double zfull) {
  const bool topk_on = top_k > 0, topp_on = top_p < 1.f;
  constexpr int kb = Elt<DT>::kKeyBits;
  uint32_t kk = 0, ck = 0, tk = 0;
  double zk = zfull;
  if (topk_on) {
    for (int bit = kb - 1; bit >= 0; --bit) {
      const uint32_t cand = kk | (1u << bit);
      if (row_pass<DT>(sh, row, V, aligned, PASS_COUNT_GE, cand, rs) >= (double)top_k) kk = cand;
    }
    const uint32_t gt = (kk == 0xFFFFFFFFu)
        ? 0u : static_cast<uint32_t>(row_pass<DT>(sh, row, V, aligned, PASS_COUNT_GE, kk + 1u, rs));
    ck = static_cast<uint32_t>(top_k) - gt;
    tk = static_cast<uint32_t>(row_pass<DT>(sh, row, V, aligned, PASS_COUNT_EQ, kk, rs));
    const float ek = lat_mass(value_of_key<DT>(kk), rs.c, rs.K);
    zk = row_pass<DT>(sh, row, V, aligned, PASS_MASS_GT, kk, rs) + (double)ck * (double)ek;
  }
  uint32_t kstar = kk, cstar = ck, tstar = tk;
  double zkept = zk;
  if (topp_on) {
    const double target = (double)top_p * zk;
    auto G = [&](uint32_t kappa) -> double {  // mass of the top-k set strictly above kappa
      if (topk_on && kappa < kk) return zk;
      return row_pass<DT>(sh, row, V, aligned, PASS_MASS_GT, kappa, rs);
    };
    uint32_t k0;
    if (G(0u) < target) {
      k0 = 0u;
    } else {
      uint32_t kp = 0u;
      for (int bit = kb - 1; bit >= 0; --bit) {
        const uint32_t cand = kp | (1u << bit);
        if (G(cand) >= target) kp = cand;
      }
      k0 = kp + 1u;
    }
    kstar = static_cast<uint32_t>(row_pass<DT>(sh, row, V, aligned, PASS_MIN_GE, k0, rs));
    const double mb = G(kstar);
    tstar = static_cast<uint32_t>(row_pass<DT>(sh, row, V, aligned, PASS_COUNT_EQ, kstar, rs));
    const uint32_t avail = (topk_on && kstar == kk) ? ck : tstar;
    const float ep = lat_mass(value_of_key<DT>(kstar), rs.c, rs.K);
    const double xneed = (target - mb) / (double)ep;
    uint32_t cp = avail;
    if (xneed < (double)avail) cp = max(1u, static_cast<uint32_t>(ceil(xneed)));
    cstar = cp;
    zkept = mb + (double)cp * (double)ep;
  }
  CutOut co;
  co.kstar = kstar;
  co.keep = cstar;
  co.total = tstar;
  co.found = 1;
  co.zkept = df_from(zkept);
  return co;
}

// ------------------------------------------------------ segments & lists

// Warp w owns vectors [seg_beg, seg_end) of a row: consecutive vectors in
// index order (iteration, lane, element).
struct Seg {
  int beg, end, iters;
};
__device__ __forceinline__ Seg warp_seg(int nvec, int warp) {
  const int vpw = ((nvec + kWarps - 1) / kWarps + 31) / 32 * 32;
  Seg s;
  s.beg = min(nvec, warp * vpw);
  s.end = min(nvec, s.beg + vpw);
  s.iters = (s.end - s.beg + 31) / 32;
  return s;
}

// List entry: element index within the warp segment (high 16 bits) and the
// element's 16-bit pattern (low 16 bits).  Lists are bf16 only.
__device__ __forceinline__ uint32_t entry_make(uint32_t local, uint32_t bits) { return (local << 16) | bits; }
__device__ __forceinline__ uint32_t entry_local(uint32_t e) { return e >> 16; }
__device__ __forceinline__ uint32_t entry_bits(uint32_t e) { return e & 0xFFFFu; }

// Keeps, in order, the entries of one warp's list whose key is at least
// kthr; returns the new length.  Whole warp.
__device__ __forceinline__ uint32_t list_purge(uint32_t* list, uint32_t len, uint32_t kthr) {
  const int lane = threadIdx.x & 31;
  uint32_t out = 0;
  for (uint32_t base = 0; base < len; base += 32) {
    const uint32_t i = base + lane;
    const uint32_t e = i < len ? list[i] : 0u;
    const bool keep = i < len && Elt<DT_BF16>::key(entry_bits(e)) >= kthr;
    const unsigned ball = __ballot_sync(kFull, keep);
    __syncwarp();
    if (keep) list[out + __popc(ball & ((1u << lane) - 1u))] = e;
    out += __popc(ball);
    __syncwarp();
  }
  return out;
}

// Tie cut from one warp-ordered set of tokens of value kstar: every warp
// counts its tokens (list entries or segment elements), the warp holding the
// keep-th one (0-based) finds its row index.  Whole CTA.
template <int DT, bool FROM_LIST>
__device__ __noinline__ int tie_cut_of(Shm& sh, const uint32_t* list, uint32_t len, const unsigned char* row, int V,
                                       bool aligned, uint32_t kstar, uint32_t keep) {
  using E = Elt<DT>;
  using H = Hot<DT>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = (V + E::kPerVec - 1) / E::kPerVec;
  const Seg sg = warp_seg(nvec, warp);
  const uint32_t thr = H::thr_pack(E::bits_of_key(kstar));
  uint32_t c = 0;
  if (FROM_LIST) {
    for (uint32_t i = lane; i < len; i += 32) c += (E::key(entry_bits(list[i])) == kstar) ? 1u : 0u;
  } else {
    for (int v = sg.beg + lane; v < sg.end; v += 32) {
      const uint4 x = load_vec<DT>(row, v, V, aligned);
      c += __popc(H::mask_eq(x, thr) & vmask<DT>(v, V));
    }
  }
  c = warp_sum_u32(c);
  if (lane == 0) sh.w_u[warp][0] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t run = 0;
    sh.tie_warp[0] = -1;
    for (int w = 0; w < kWarps; ++w) {
      if (run + sh.w_u[w][0] > keep) { sh.tie_warp[0] = w; sh.tie_j[0] = keep - run; break; }
      run += sh.w_u[w][0];
    }
    sh.tie_cut[0] = V;  // all kept (only if the counts disagree)
  }
  __syncthreads();
  if (warp == sh.tie_warp[0]) {
    uint32_t jj = sh.tie_j[0];
    const int seg_lo = sg.beg * E::kPerVec;
    const int rounds = FROM_LIST ? static_cast<int>((len + 31) / 32) : sg.iters;
    for (int it = 0; it < rounds; ++it) {
      uint32_t msk = 0u;
      int base_idx = 0;
      if (FROM_LIST) {
        const uint32_t i = it * 32 + lane;
        if (i < len && E::key(entry_bits(list[i])) == kstar) {
          msk = 1u;
          base_idx = seg_lo + static_cast<int>(entry_local(list[i]));
        }
      } else {
        const int v = sg.beg + it * 32 + lane;
        if (v < sg.end) msk = H::mask_eq(load_vec<DT>(row, v, V, aligned), thr) & vmask<DT>(v, V);
        base_idx = v * E::kPerVec;
      }
      const uint32_t cc = __popc(msk);
      const uint32_t incl = warp_incl_scan_u32(cc);
      const uint32_t tot = __shfl_sync(kFull, incl, 31);
      if (jj < tot) {
        if (incl > jj && incl - cc <= jj) {
          uint32_t mm = msk;
          for (uint32_t q = jj - (incl - cc); q > 0; --q) mm &= mm - 1u;
          sh.tie_cut[0] = FROM_LIST ? base_idx : base_idx + (__ffs(mm) - 1);
        }
        break;
      }
      jj -= tot;
    }
  }
  __syncthreads();
  const int r = sh.tie_cut[0];
  __syncthreads();
  return r;
}

// The filtered, normalised probabilities of a row, written out.
template <int DT>
__device__ __noinline__ void write_probs(const unsigned char* row, int V, bool aligned, const RowStat& rp,
                                         float* out) {
  using E = Elt<DT>;
  const int nvec = (V + E::kPerVec - 1) / E::kPerVec;
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    const uint4 x = load_vec<DT>(row, v, V, aligned);
#pragma unroll
    for (int j = 0; j < E::kPerVec; ++j) {
      const int t = v * E::kPerVec + j;
      if (t < V) out[t] = rp.bad ? 0.f : prob_of<DT>(rp, E::bits_of(x, j), t);
    }
  }
}

// Draw weight of token j: max(0, p - q) (residual) or p (bonus / degenerate).
template <int DT>
__device__ __forceinline__ float weight_of(const RowStat& rp, const RowStat& rq, uint32_t bp, const unsigned char* rowq,
                                           int j, bool use_q, float* pv_out) {
  const float pv = prob_of<DT>(rp, bp, j);
  *pv_out = pv;
  if (!use_q || pv == 0.f) return pv;
  const float qv = prob_of<DT>(rq, Elt<DT>::bits_at(rowq, j), j);
  return fmaxf(pv - qv, 0.f);
}

}  // namespace

// One unit (b, pos) with NR rows (2: target and draft, 1: target only).
template <int DT, int NR>
__device__ __forceinline__ void unit_body(const SampleArgs& a, Shm& sh, uint32_t* lists, uint32_t* hist, int unit, int b,
                                          int pos, const unsigned char* rowp, const unsigned char* rowq) {
  using E = Elt<DT>;
  using H = Hot<DT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;
  const float T = a.temperature_per_seq ? a.temperature_per_seq[b] : a.temperature;
  const bool bad_t = !(T > 0.f) || isinf(T);
  const float c = kLog2e / T;
  const u64 c2 = pkf(c, c);
  const int nvec = (V + E::kPerVec - 1) / E::kPerVec;
  const Seg sg = warp_seg(nvec, warp);
  const unsigned char* rows[2] = {rowp, rowq};
  const bool aligned[2] = {a.aligned_target != 0, a.aligned_draft != 0};
  const bool topk_on = a.top_k > 0;
  const bool topp_on = a.top_p < 1.f;
  const bool filt = topk_on || topp_on;
  // candidate lists: bf16 rows with a cut, segments short enough to index
  const bool use_lists = DT == DT_BF16 && filt && !bad_t && (sg.end - sg.beg) * E::kPerVec <= (1 << kSegBits) &&
                         ((nvec + kWarps - 1) / kWarps + 31) / 32 * 32 * E::kPerVec <= (1 << kSegBits);
  const float dtheta = kTheta / c;  // kTheta octaves of mass, in logit units
  uint32_t* wl[2] = {lists + (0 * kWarps + warp) * kListCap, lists + (1 * kWarps + warp) * kListCap};

  if (filt)
    for (int t = tid; t < NR * kWindow; t += kThreads) hist[t] = 0u;
  __syncthreads();

  // --------------------------------------------------- phase 1: stream
  float mt[NR];             // thread maximum
  int kt[NR];               // thread lattice exponent
  u64 acc0[NR], acc1[NR];   // thread sums of 2^(l c - kt)
  float mw[NR];             // running maximum known to the warp (uniform)
  uint32_t len[NR];         // list lengths (uniform)
  uint32_t kthr[NR];        // current list bound, as a key (uniform)
  uint32_t kfloor[NR];      // raised bound: the list is complete above it
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    mt[r] = -INFINITY;
    kt[r] = -(1 << 30);
    acc0[r] = 0ull;
    acc1[r] = 0ull;
    mw[r] = -INFINITY;
    len[r] = 0u;
    kthr[r] = 0u;
    kfloor[r] = 0u;
  }
  // every warp runs the same number of iterations (the CTA barriers below)
  const int iters_all = (((nvec + kWarps - 1) / kWarps + 31) / 32 * 32) / 32;
  for (int it = 0; it < iters_all; it += 2) {
    const int v0 = sg.beg + it * 32 + lane;
    const int v1 = v0 + 32;
    uint4 x[NR][2];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      x[r][0] = v0 < sg.end ? load_vec<DT>(rows[r], v0, V, aligned[r]) : make_uint4(H::kPad, H::kPad, H::kPad, H::kPad);
      x[r][1] = v1 < sg.end ? load_vec<DT>(rows[r], v1, V, aligned[r]) : make_uint4(H::kPad, H::kPad, H::kPad, H::kPad);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      float vm[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        vm[u] = H::vmax(x[r][u]);
        const float L = vm[u] * c;
        if (L > static_cast<float>(kt[r]) && L < 1073741824.f) {  // raise the lattice exponent (rare)
          const int knew = static_cast<int>(ceilf(L));
          const float s = exp2i(kt[r] - knew);
          acc0[r] = mul2(acc0[r], pkf(s, s));
          acc1[r] = mul2(acc1[r], pkf(s, s));
          kt[r] = knew;
        }
        const float nk = -static_cast<float>(kt[r]);
        H::mass_vec(x[r][u], c2, pkf(nk, nk), acc0[r], acc1[r]);
        mt[r] = max_nan(mt[r], vm[u]);
      }
      if (use_lists) {
        // the bound: kTheta octaves below the running maximum (at most the
        // row maximum), never below the raised floor
        const float m_new = warp_max_nan(max_nan(vm[0], vm[1]));
        if (m_new > mw[r]) mw[r] = m_new;
        {
          const float tv = mw[r] - dtheta;
          const uint32_t kb = tv > -3.0e38f ? E::key(bits_round_down<DT>(tv)) : 0u;
          kthr[r] = max(kfloor[r], kb);
        }
        // candidates: elements at or above the bound, appended in index order
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int v = v0 + 32 * u;
          for (;;) {
            const float thr_v = value_of_key<DT>(kthr[r]);
            const bool any = v < sg.end && vm[u] >= thr_v;
            if (__ballot_sync(kFull, any) == 0u) break;
            const uint32_t msk = any ? (H::mask_ge(x[r][u], H::thr_pack(E::bits_of_key(kthr[r]))) & vmask<DT>(v, V)) : 0u;
            const uint32_t cnt = __popc(msk);
            const uint32_t incl = warp_incl_scan_u32(cnt);
            const uint32_t tot = __shfl_sync(kFull, incl, 31);
            if (len[r] + tot > static_cast<uint32_t>(kListCap)) {
              len[r] = list_purge(wl[r], len[r], kthr[r]);
              if (len[r] + tot > static_cast<uint32_t>(kListCap)) {
                // still full: raise the floor (a step toward the warp maximum)
                const uint32_t kmw = key_of_float<DT>(mw[r]);
                const uint32_t step = kmw > kthr[r] ? max(1u, (kmw - kthr[r]) / 8u) : 1u;
                kfloor[r] = kthr[r] + step;
                kthr[r] = kfloor[r];
                continue;
              }
            }
            uint32_t pos_w = len[r] + incl - cnt;
            uint32_t mm = msk;
            while (mm) {
              const int j = __ffs(mm) - 1;
              mm &= mm - 1u;
              wl[r][pos_w++] = entry_make(static_cast<uint32_t>((v - sg.beg) * 8 + j), E::bits_of(x[r][u], j));
            }
            len[r] += tot;
            break;
          }
        }
      }
    }
    if (use_lists && ((it >> 1) % kSyncEvery) == kSyncEvery - 1) {
      // share the running maxima across the CTA (fixed points: deterministic)
      const int slot = ((it >> 1) / kSyncEvery) & 1;
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < NR; ++r) sh.x_m[slot][warp][r] = mw[r];
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        float mm = mw[r];
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, sh.x_m[slot][w][r]);
        mw[r] = mm;
      }
    }
  }
  __syncwarp();

  // ------------------------------------------ phase 2: row maximum and sum
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float s0, s1, s2, s3;
    upk(acc0[r], s0, s1);
    upk(acc1[r], s2, s3);
    float zt = (s0 + s1) + (s2 + s3);
    const int kw = warp_max_i32(kt[r]);
    zt *= exp2i(kt[r] - kw);
    zt = warp_sum_f32(zt);
    const float mx = warp_max_nan(mt[r]);
    if (lane == 0) {
      sh.w_m[warp][r] = mx;
      sh.w_k[warp][r] = kw;
      sh.w_z[warp][r] = zt;
      sh.w_n[warp][r] = len[r];
      sh.w_floor[warp][r] = kfloor[r];
    }
  }
  __syncthreads();
  float m[NR], K[NR];
  bool bad[NR], cov[NR];
  bool any_bad = bad_t;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float mx = -INFINITY;
    int kk = -(1 << 30);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      mx = max_nan(mx, sh.w_m[w][r]);
      kk = max(kk, sh.w_k[w][r]);
    }
    DF z{0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kWarps; ++w) z = df_add(z, sh.w_z[w][r] * exp2i(sh.w_k[w][r] - kk));
    m[r] = mx;
    K[r] = static_cast<float>(kk);
    // the lattice exponent must stay an int: |max| log2(e) / T < 2^30
    bad[r] = bad_t || !isfinite(mx) || !(fabsf(mx * c) < 1073741824.f);
    any_bad |= bad[r];
    cov[r] = use_lists;
    if (tid == 0) sh.z[r] = z;
  }

  if (any_bad) {
    if (a.mode == MODE_PROBS) {
      float* out = a.out_probs + static_cast<size_t>(unit) * V;
      for (int t = tid; t < V; t += kThreads) out[t] = 0.f;
      if (tid == 0) set_status(a.status, SPEC_STATUS_BAD_ROW);
    } else if (tid == 0) {
      const int kq = a.k;
      UnitRec* rec = a.recs + unit;
      uint32_t add = 1u;
      uint32_t st = SPEC_STATUS_BAD_ROW;
      rec->drawn = -1;
      if (NR == 2) {
        const int x = a.tokens[static_cast<size_t>(b) * kq + pos];
        if (!(x >= 0 && x < V)) st |= SPEC_STATUS_BAD_TOKEN;
        rec->accept = 0;
        rec->px = 0.f;
        rec->qx = 0.f;
        if (a.out_p) a.out_p[static_cast<size_t>(b) * kq + pos] = 0.f;
        if (a.out_q) a.out_q[static_cast<size_t>(b) * kq + pos] = 0.f;
        add = 2u;
      }
      set_status(a.status, st);
      __threadfence();
      const uint32_t before = atomicAdd(a.tickets + b, add);
      if (before + add == static_cast<uint32_t>(2 * kq + 1)) sample_finalize(a, b);
    }
    return;
  }

  // --------------------------- phase 3: histogram of the candidates' values
  // Every element within kTheta octaves of the row maximum (key >= klo) is
  // on a list; the histogram covers keys klo .. kmax (at most kWindow).
  uint32_t klo[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const uint32_t kmax = key_of_float<DT>(m[r]);
    const float tv = m[r] - dtheta;
    uint32_t kl = tv > -3.0e38f ? E::key(bits_round_up<DT>(tv)) : 0u;
    const uint32_t gtop = kmax >> 2;
    if (gtop >= static_cast<uint32_t>(kGroups - 1)) kl = max(kl, 4u * (gtop - static_cast<uint32_t>(kGroups - 1)));
    for (int w = 0; w < kWarps; ++w) kl = max(kl, sh.w_floor[w][r]);  // every list is complete above kl
    klo[r] = kl;
    if (cov[r]) {
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t n_w = sh.w_n[w][r];
        const uint32_t* lw = lists + (r * kWarps + w) * kListCap;
        for (uint32_t i = tid; i < n_w; i += kThreads) {
          const uint32_t k = E::key(entry_bits(lw[i]));
          if (k >= kl) red_add_shared(smem_addr(hist + r * kWindow + (k & kSlotMask)), 1u);
        }
      }
    }
  }
  if (tid < 2) { sh.cut[tid].found = 0; sh.cutk[tid].found = 0; }
  __syncthreads();

  // ---------------------------------------------- phase 4: the cut scan
  if (filt) {
    const int r_s = (NR == 2) ? (warp >> 2) : 0;
    const int wq = warp & (kScanWarps - 1);
    const bool scanner = ((NR == 2) || warp < kScanWarps) && (r_s == 0 ? cov[0] : cov[NR - 1]);
    const float m_s = r_s == 0 ? m[0] : m[NR - 1];
    const float K_s = r_s == 0 ? K[0] : K[NR - 1];
    const uint32_t klo_s = r_s == 0 ? klo[0] : klo[NR - 1];
    const uint32_t kmax_s = key_of_float<DT>(m_s);
    uint32_t cnt[4] = {0u, 0u, 0u, 0u}, top = 0u, Cl = 0u, Cex = 0u;
    float ms[4] = {0.f, 0.f, 0.f, 0.f}, Ml = 0.f;
    DF Mex{0.f, 0.f};
    bool valid = false;
    if (scanner) {
      const uint32_t gtop = kmax_s >> 2;
      const uint32_t gi = static_cast<uint32_t>(wq * 32 + lane);
      if (gi <= gtop) {
        const uint32_t grp = gtop - gi;
        top = 4u * grp + 3u;
        if (top >= klo_s) {
          valid = true;
          const uint4 h4 = lds128(smem_addr(hist + r_s * kWindow + 4u * (grp & static_cast<uint32_t>(kGroups - 1))));
          const uint32_t hv[4] = {h4.w, h4.z, h4.y, h4.x};  // keys top, top-1, top-2, top-3
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t key = top - static_cast<uint32_t>(j);
            const uint32_t s = (key > kmax_s || key < klo_s) ? 0u : hv[j];
            cnt[j] = s;
            ms[j] = s ? lat_mass(value_of_key<DT>(key), c, K_s) : 0.f;
            Cl += s;
            Ml += static_cast<float>(s) * ms[j];
          }
        }
      }
      const uint32_t Cin = warp_incl_scan_u32(Cl);
      const DF Min = warp_incl_scan_df(DF{Ml, 0.f});
      Cex = Cin - Cl;
      Mex = df_shfl_up(Min, 1);
      if (lane == 0) Mex = DF{0.f, 0.f};
      if (lane == 31) {
        sh.s_C[r_s][wq] = Cin;
        sh.s_M[r_s][wq] = Min;
      }
    }
    __syncthreads();
    uint32_t offC = 0u;
    DF offM{0.f, 0.f}, nxtM{0.f, 0.f}, totM{0.f, 0.f};
    if (scanner) {
#pragma unroll
      for (int q = 0; q < kScanWarps; ++q) {
        const uint32_t cq = sh.s_C[r_s][q];
        const DF mq = sh.s_M[r_s][q];
        if (q < wq) { offC += cq; offM = df_add2(offM, mq); }
        if (q <= wq) nxtM = df_add2(nxtM, mq);
        totM = df_add2(totM, mq);
      }
    }
    if (topk_on && scanner) {  // the value where the running count reaches top_k
      const uint32_t Kc = static_cast<uint32_t>(a.top_k);
      const uint32_t wC = sh.s_C[r_s][wq];
      if (offC < Kc && offC + wC >= Kc) {
        const uint32_t cb = offC + Cex;
        const unsigned ball = __ballot_sync(kFull, valid && cb < Kc);
        const int l = 31 - __clz(ball | 1u);
        if (lane == l && valid && cb < Kc) {
          uint32_t run = cb;
          DF mb = df_add2(offM, Mex);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (run < Kc && run + cnt[j] >= Kc) {
              CutOut co;
              co.kstar = top - static_cast<uint32_t>(j);
              co.keep = Kc - run;
              co.total = cnt[j];
              co.found = 1;
              co.zkept = df_add(mb, static_cast<float>(Kc - run) * ms[j]);
              sh.cutk[r_s] = co;
              if (!topp_on) sh.cut[r_s] = co;
            }
            run += cnt[j];
            mb = df_add(mb, static_cast<float>(cnt[j]) * ms[j]);
          }
        }
      }
    }
    if (topk_on && topp_on) __syncthreads();
    if (topp_on && scanner) {  // a token is kept while the mass ranked before it is below top_p * Z
      const CutOut ck = sh.cutk[r_s];
      if (!topk_on || ck.found) {
        const DF target = df_mul_f(topk_on ? ck.zkept : sh.z[r_s], a.top_p);
        const bool wlast = !df_lt(totM, target) && df_lt(offM, target) &&
                           (wq == kScanWarps - 1 || !df_lt(nxtM, target));
        if (wlast) {
          const DF mbl = df_add2(offM, Mex);
          const unsigned ball = __ballot_sync(kFull, valid && df_lt(mbl, target));
          const int l = 31 - __clz(ball | 1u);
          if (lane == l && valid && df_lt(mbl, target)) {
            DF mb = mbl, mb_last{0.f, 0.f};
            int jl = -1;
            uint32_t cl = 0u;
            bool done = false;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t key = top - static_cast<uint32_t>(j);
              uint32_t ce = cnt[j];
              if (topk_on) ce = key < ck.kstar ? 0u : (key == ck.kstar ? ck.keep : ce);
              if (!done && ce > 0u) {
                const DF after = df_add(mb, static_cast<float>(ce) * ms[j]);
                jl = j;
                cl = ce;
                mb_last = mb;
                if (!df_lt(after, target)) {
                  const float need = df_float(df_add(target, -mb.hi)) - mb.lo;
                  uint32_t keep = static_cast<uint32_t>(ceilf(need / ms[j]));
                  keep = max(1u, min(keep, ce));
                  CutOut co;
                  co.kstar = key;
                  co.keep = keep;
                  co.total = cnt[j];
                  co.found = 1;
                  co.zkept = df_add(mb, static_cast<float>(keep) * ms[j]);
                  sh.cut[r_s] = co;
                  done = true;
                }
                mb = after;
              }
            }
            if (!done && jl >= 0) {  // rounding put the crossing past this lane: all of its last value
              CutOut co;
              co.kstar = top - static_cast<uint32_t>(jl);
              co.keep = cl;
              co.total = cnt[jl];
              co.found = 1;
              co.zkept = df_add(mb_last, static_cast<float>(cl) * ms[jl]);
              sh.cut[r_s] = co;
            }
          }
        }
      }
    }
    __syncthreads();
  }

  // ------------------------------------ phase 5: kept set of each row
#pragma unroll 1
  for (int r = 0; r < NR; ++r) {
    RowStat rs;
    rs.c = c;
    rs.K = r == 0 ? K[0] : K[NR - 1];
    rs.m = r == 0 ? m[0] : m[NR - 1];
    rs.kmax = key_of_float<DT>(rs.m);
    rs.bad = 0;
    rs.all_kept = filt ? 0 : 1;
    rs.covered = (r == 0 ? cov[0] : cov[NR - 1]) ? 1 : 0;
    rs.kstar = 0u;
    rs.tie_cut = V;
    float zk = df_float(sh.z[r]);
    if (filt) {
      CutOut co = sh.cut[r];
      const bool from_lists = co.found != 0;
      if (!from_lists) {
        rs.covered = 0;
        co = search_cut<DT>(sh, rows[r], V, aligned[r], a.top_k, a.top_p, rs, df_double(sh.z[r]));
      }
      rs.kstar = co.kstar;
      zk = df_float(co.zkept);
      if (co.keep < co.total) {
        const uint32_t* lw = lists + (r * kWarps + warp) * kListCap;
        rs.tie_cut = from_lists
            ? tie_cut_of<DT, true>(sh, lw, sh.w_n[warp][r], rows[r], V, aligned[r], co.kstar, co.keep)
            : tie_cut_of<DT, false>(sh, lw, 0u, rows[r], V, aligned[r], co.kstar, co.keep);
      }
    }
    rs.zkept = zk;
    rs.inv_z = 1.f / zk;
    if (tid == 0) sh.rs[r] = rs;
  }
  __syncthreads();
  const RowStat rp = sh.rs[0];
  const RowStat rq = sh.rs[NR - 1];

  if (a.mode == MODE_PROBS) {
    write_probs<DT>(rows[0], V, aligned[0], rp, a.out_probs + static_cast<size_t>(unit) * V);
    return;
  }

  const int kq = a.k;
  // ------------------------------------- phase 6: accept test at x_pos
  if (NR == 2 && tid == 0) {
    const int x = a.tokens[static_cast<size_t>(b) * kq + pos];
    UnitRec* rec = a.recs + unit;
    float px = 0.f, qx = 0.f;
    if (x >= 0 && x < V) {
      px = prob_of<DT>(rp, E::bits_at(rows[0], x), x);
      qx = prob_of<DT>(rq, E::bits_at(rows[NR - 1], x), x);
      const float u = a.uniforms[static_cast<size_t>(b) * (kq + 2) + pos];
      rec->accept = (u * qx < px) ? 1 : 0;
    } else {
      rec->accept = 0;
      set_status(a.status, SPEC_STATUS_BAD_TOKEN);
    }
    rec->px = px;
    rec->qx = qx;
    if (a.out_p) a.out_p[static_cast<size_t>(b) * kq + pos] = px;
    if (a.out_q) a.out_q[static_cast<size_t>(b) * kq + pos] = qx;
    __threadfence();
    if (atomicAdd(a.tickets + b, 1u) == static_cast<uint32_t>(2 * kq)) sample_finalize(a, b);
  }

  // ------------- phase 7: residual (or bonus) by warps, in index order
  // On the fast path each warp walks its list of p (the kept set of p is on
  // it); otherwise its segment of the row.
  const bool lists_p = rp.covered && !rp.all_kept;
  const uint32_t* lp = lists + (0 * kWarps + warp) * kListCap;
  const uint32_t np = lists_p ? sh.w_n[warp][0] : 0u;
  const int seg_lo = sg.beg * E::kPerVec;
  {
    float s = 0.f, sp = 0.f;
    if (lists_p) {
      for (uint32_t i = lane; i < np; i += 32) {
        const uint32_t e = lp[i];
        const int j = seg_lo + static_cast<int>(entry_local(e));
        float pv;
        s += weight_of<DT>(rp, rq, entry_bits(e), rows[NR - 1], j, NR == 2, &pv);
        sp += pv;
      }
    } else {
      for (int v = sg.beg + lane; v < sg.end; v += 32) {
        const uint4 xp = load_vec<DT>(rows[0], v, V, aligned[0]);
        const uint4 xq = NR == 2 ? load_vec<DT>(rows[NR - 1], v, V, aligned[NR - 1]) : xp;
#pragma unroll
        for (int j = 0; j < E::kPerVec; ++j) {
          const int t = v * E::kPerVec + j;
          if (t < V) {
            const float pv = prob_of<DT>(rp, E::bits_of(xp, j), t);
            sp += pv;
            s += NR == 2 ? fmaxf(pv - (pv > 0.f ? prob_of<DT>(rq, E::bits_of(xq, j), t) : 0.f), 0.f) : pv;
          }
        }
      }
    }
    s = warp_sum_f32(s);
    sp = warp_sum_f32(sp);
    if (lane == 0) {
      sh.w_s[warp] = s;
      sh.w_sp[warp] = sp;
    }
  }
  __syncthreads();
  if (tid == 0) {
    DF S{0.f, 0.f}, Sp{0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      S = df_add(S, sh.w_s[w]);
      Sp = df_add(Sp, sh.w_sp[w]);
    }
    bool use_q = NR == 2;
    const float* ws = sh.w_s;
    if (NR == 2 && !(S.hi > 0.f)) {  // degenerate residual: draw from p instead
      use_q = false;
      S = Sp;
      ws = sh.w_sp;
    }
    const float u_draw = a.uniforms[static_cast<size_t>(b) * (kq + 2) + (NR == 2 ? kq + 1 : kq)];
    const DF target = df_mul_f(S, u_draw);
    DF run{0.f, 0.f}, base{0.f, 0.f}, lbase{0.f, 0.f};
    int wsel = -1, wlast = -1;
    for (int w = 0; w < kWarps; ++w) {
      const float sw = ws[w];
      const DF nxt = df_add(run, sw);
      if (sw > 0.f) { wlast = w; lbase = run; }
      if (wsel < 0 && sw > 0.f && df_lt(target, nxt)) { wsel = w; base = run; }
      run = nxt;
    }
    if (wsel < 0) { wsel = wlast; base = lbase; }
    sh.draw_warp = use_q ? wsel : -2 - wsel;  // -2 - w: weights are p
    sh.draw_base = df_float(df_add2(target, df_neg(base)));
  }
  __syncthreads();
  const int dw = sh.draw_warp;
  const bool use_q = dw >= 0;
  const int wsel = use_q ? dw : -2 - dw;
  if (warp == wsel) {
    const float tw = sh.draw_base;
    float run = 0.f;
    int token = -1, last_pos = -1;
    const int rounds = lists_p ? static_cast<int>((np + 31) / 32) : sg.iters;
    for (int it = 0; it < rounds && token < 0; ++it) {
      float w[8];
      int idx[8];
      float ls = 0.f;
      int lpos = -1;
#pragma unroll
      for (int j = 0; j < 8; ++j) { w[j] = 0.f; idx[j] = -1; }
      if (lists_p) {
        const uint32_t i = it * 32 + lane;
        if (i < np) {
          const uint32_t e = lp[i];
          float pv;
          idx[0] = seg_lo + static_cast<int>(entry_local(e));
          w[0] = weight_of<DT>(rp, rq, entry_bits(e), rows[NR - 1], idx[0], use_q, &pv);
        }
      } else {
        const int v = sg.beg + it * 32 + lane;
        if (v < sg.end) {
          const uint4 xp = load_vec<DT>(rows[0], v, V, aligned[0]);
          const uint4 xq = use_q ? load_vec<DT>(rows[NR - 1], v, V, aligned[NR - 1]) : xp;
#pragma unroll
          for (int j = 0; j < E::kPerVec; ++j) {
            const int t = v * E::kPerVec + j;
            if (t < V) {
              const float pv = prob_of<DT>(rp, E::bits_of(xp, j), t);
              w[j] = use_q ? fmaxf(pv - (pv > 0.f ? prob_of<DT>(rq, E::bits_of(xq, j), t) : 0.f), 0.f) : pv;
              idx[j] = t;
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        ls += w[j];
        if (w[j] > 0.f) lpos = idx[j];
      }
      const float incl = warp_incl_scan(ls);
      const unsigned ball = __ballot_sync(kFull, ls > 0.f && run + incl > tw);
      const int lastl = 31 - __clz(__ballot_sync(kFull, lpos >= 0) | 1u);
      const int lp2 = __shfl_sync(kFull, lpos, lastl);
      if (lp2 >= 0) last_pos = lp2;
      if (ball) {
        const int l = __ffs(ball) - 1;
        int tok = -1;
        if (lane == l) {
          float cum = run + (incl - ls);
          int lastj = -1;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (w[j] > 0.f) lastj = idx[j];
            cum += w[j];
            if (tok < 0 && w[j] > 0.f && cum > tw) tok = idx[j];
          }
          if (tok < 0) tok = lastj;
        }
        token = __shfl_sync(kFull, tok, l);
      }
      run += __shfl_sync(kFull, incl, 31);
    }
    if (token < 0) token = last_pos;  // only reachable through rounding
    if (lane == 0) {
      a.recs[unit].drawn = token;
      __threadfence();
      if (atomicAdd(a.tickets + b, 1u) == static_cast<uint32_t>(2 * kq)) sample_finalize(a, b);
    }
  } else if (wsel < 0 && tid == 0) {  // nothing to draw from (all mass rounded away)
    a.recs[unit].drawn = -1;
    __threadfence();
    if (atomicAdd(a.tickets + b, 1u) == static_cast<uint32_t>(2 * kq)) sample_finalize(a, b);
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 4) sample_kernel(const SampleArgs a) {
  using E = Elt<DT>;
  const int unit = static_cast<int>(blockIdx.x);
  const int V = a.V;
  __shared__ Shm sh;
  extern __shared__ __align__(16) uint32_t dsm[];
  uint32_t* lists = dsm;                                // [2][kWarps][kListCap]
  uint32_t* hist = dsm + 2 * kWarps * kListCap;         // [2][kWindow]
  if (a.mode == MODE_SAMPLE) {
    const int b = unit / (a.k + 1);
    const int pos = unit % (a.k + 1);
    const unsigned char* rowp =
        static_cast<const unsigned char*>(a.target) + static_cast<size_t>(unit) * V * E::kBytes;
    if (pos < a.k) {
      const unsigned char* rowq = static_cast<const unsigned char*>(a.draft) +
                                  (static_cast<size_t>(b) * a.k + pos) * static_cast<size_t>(V) * E::kBytes;
      unit_body<DT, 2>(a, sh, lists, hist, unit, b, pos, rowp, rowq);
    } else {
      unit_body<DT, 1>(a, sh, lists, hist, unit, b, pos, rowp, rowp);
    }
  } else {
    const unsigned char* rowp =
        static_cast<const unsigned char*>(a.target) + static_cast<size_t>(unit) * V * E::kBytes;
    unit_body<DT, 1>(a, sh, lists, hist, unit, unit, 0, rowp, rowp);
  }
}

// The last writer of sequence b applies the first-rejection rule and commits.
__device__ void sample_finalize(const SampleArgs& a, int b) {
  __threadfence();
  const int k = a.k;
  const UnitRec* rec = a.recs + static_cast<size_t>(b) * (k + 1);
  int n = k;
  for (int i = 0; i < k; ++i) {
    if (__ldcg(&rec[i].accept) == 0) { n = i; break; }
  }
  int32_t* out = a.out_tokens + static_cast<size_t>(b) * (k + 1);
  for (int i = 0; i < n; ++i) out[i] = a.tokens[static_cast<size_t>(b) * k + i];
  out[n] = __ldcg(&rec[n].drawn);
  for (int i = n + 1; i <= k; ++i) out[i] = -1;
  a.out_n[b] = n;
  // leave the workspace zeroed for the next call, whatever its shape
  UnitRec* wrec = a.recs + static_cast<size_t>(b) * (k + 1);
  for (int i = 0; i <= k; ++i) wrec[i] = UnitRec{0, 0, 0.f, 0.f};
  a.tickets[b] = 0u;
}

// ------------------------------------------------------------------ launch

size_t sample_smem_bytes(int dtype, bool filter) {
  (void)dtype;
  return filter ? (2 * kWarps * kListCap + 2 * kWindow) * sizeof(uint32_t) : 16;
}

template <int DT>
static int launch_one(const SampleArgs& a, int units, size_t smem, cudaStream_t st) {
  auto kern = sample_kernel<DT>;
  static size_t configured = 0;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  kern<<<units, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

int launch_sample(const SampleArgs& a, int dtype, int units, void* stream) {
  const bool filter = a.top_k > 0 || a.top_p < 1.f;
  const size_t smem = sample_smem_bytes(dtype, filter);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == DT_BF16) return launch_one<DT_BF16>(a, units, smem, st);
  if (dtype == DT_F32) return launch_one<DT_F32>(a, units, smem, st);
  return cudaErrorInvalidValue;
}

}  // namespace specv
