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
// How (one GPU, memory-bound): a thread-block cluster of CS CTAs owns one
// unit (b, i).  Each CTA bulk-copies (TMA, cp.async.bulk) its 1/CS slice of
// the target row and of the draft row into shared memory, so every logit is
// read from HBM exactly once.  Row statistics are combined across the
// cluster through distributed shared memory:
//   1. the row maximum (packed bf16x2 max over shared memory);
//   2. the sum of masses exp((l - m) / T) (packed f32x2 arithmetic), when a
//      top-p cut needs it;
//   3. for a top-k / top-p cut, a histogram of exact values counting only
//      the tokens that can survive the cut (at most 1024 distinct values
//      below the maximum; with top-p only, also no token whose mass is below
//      (1 - top_p) * Z / V, which cannot be kept); bin masses are count x
//      mass, so the cut, its tie count and the kept normaliser come from a
//      short scan over the bins.  A cut outside the histogram (flat rows,
//      fp32 rows) falls back to an exact bitwise search over the keys.
// The accept test is done by the CTA that holds x_i; the residual (or bonus)
// inverse-CDF draw is done speculatively for every unit, so no row is read
// twice; vectors with no kept token are skipped with one packed compare.  The
// CTA that holds the drawn token writes it.  The last writer of a sequence
// (atomic ticket, no spin-wait) applies the first-rejection rule and commits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "device_common.cuh"

namespace specv {

__device__ void sample_finalize(const SampleArgs& a, int b);

namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
using u64 = unsigned long long;

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
__device__ __forceinline__ u64 sub2(u64 a, u64 b) {
  u64 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
  u64 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ u64 add2(u64 a, u64 b) {
  u64 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// 2^x for both halves: the masses of two elements, (l - m) * log2(e) / T
__device__ __forceinline__ u64 mass2(u64 l2, u64 m2, u64 c2) {
  float x, y;
  upk(mul2(sub2(l2, m2), c2), x, y);
  return pkf(ex2_approx(x), ex2_approx(y));
}

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
__device__ __forceinline__ DF df_shfl_up(DF a, int o) {
  return DF{__shfl_up_sync(kFull, a.hi, o), __shfl_up_sync(kFull, a.lo, o)};
}
__device__ __forceinline__ DF df_shfl(DF a, int l) { return DF{__shfl_sync(kFull, a.hi, l), __shfl_sync(kFull, a.lo, l)}; }
// inclusive warp prefix sum of double-floats
__device__ __forceinline__ DF warp_incl_scan_df(DF v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF w = df_shfl_up(v, o);
    if (lane >= o) v = df_add2(v, w);
  }
  return v;
}
// (a - b) rounded to float
__device__ __forceinline__ float df_diff(DF a, DF b) { return (a.hi - b.hi) + (a.lo - b.lo); }
__device__ __forceinline__ double df_value(DF a) { return static_cast<double>(a.hi) + static_cast<double>(a.lo); }

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// ------------------------------------------------- per-dtype vector kernels

template <int DT>
struct Hot;

template <>
struct Hot<DT_BF16> {
  using E = Elt<DT_BF16>;
  struct MaxAcc {
    __nv_bfloat162 a;
  };
  __device__ static __forceinline__ __nv_bfloat162 b2(uint32_t w) {
    __nv_bfloat162 r;
    *reinterpret_cast<uint32_t*>(&r) = w;
    return r;
  }
  __device__ static __forceinline__ void max_init(MaxAcc& s) { s.a = b2(0xFF80FF80u); }
  __device__ static __forceinline__ void max_vec(const uint4& v, MaxAcc& s) {
    s.a = __hmax2_nan(__hmax2_nan(s.a, b2(v.x)), __hmax2_nan(b2(v.y), __hmax2_nan(b2(v.z), b2(v.w))));
  }
  __device__ static __forceinline__ float max_finish(const MaxAcc& s) {
    return max_nan(__low2float(s.a), __high2float(s.a));
  }
  // accumulate the masses of the 8 elements into acc (two running sums)
  __device__ static __forceinline__ void mass_vec(const uint4& v, u64 m2, u64 c2, u64& acc) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) acc = add2(acc, mass2(pk2(w[i] << 16, w[i] & 0xFFFF0000u), m2, c2));
  }
  // threshold as a packed pair of one bf16 value
  __device__ static __forceinline__ uint32_t thr_pack(uint32_t bits) { return bits | (bits << 16); }
  __device__ static __forceinline__ bool any_ge(const uint4& v, uint32_t thr) {
    const __nv_bfloat162 t = b2(thr);
    return (__hge2_mask(b2(v.x), t) | __hge2_mask(b2(v.y), t) | __hge2_mask(b2(v.z), t) |
            __hge2_mask(b2(v.w), t)) != 0u;
  }
  __device__ static __forceinline__ uint32_t mask_ge(const uint4& v, uint32_t thr) {
    const __nv_bfloat162 t = b2(thr);
    const uint32_t m0 = __hge2_mask(b2(v.x), t), m1 = __hge2_mask(b2(v.y), t);
    const uint32_t m2 = __hge2_mask(b2(v.z), t), m3 = __hge2_mask(b2(v.w), t);
    return (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) | ((m2 & 1u) << 4) |
           ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u);
  }
  // bit j set iff element j equals the threshold value (-0 == +0)
  __device__ static __forceinline__ uint32_t mask_eq(const uint4& v, uint32_t thr) {
    const __nv_bfloat162 t = b2(thr);
    const uint32_t m0 = __heq2_mask(b2(v.x), t), m1 = __heq2_mask(b2(v.y), t);
    const uint32_t m2 = __heq2_mask(b2(v.z), t), m3 = __heq2_mask(b2(v.w), t);
    return (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) | ((m2 & 1u) << 4) |
           ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u);
  }
  __device__ static __forceinline__ bool any_eq(const uint4& v, uint32_t thr) {
    const __nv_bfloat162 t = b2(thr);
    return (__heq2_mask(b2(v.x), t) | __heq2_mask(b2(v.y), t) | __heq2_mask(b2(v.z), t) |
            __heq2_mask(b2(v.w), t)) != 0u;
  }
};

template <>
struct Hot<DT_F32> {
  using E = Elt<DT_F32>;
  struct MaxAcc {
    float a;
  };
  __device__ static __forceinline__ void max_init(MaxAcc& s) { s.a = -INFINITY; }
  __device__ static __forceinline__ void max_vec(const uint4& v, MaxAcc& s) {
    s.a = max_nan(max_nan(s.a, __uint_as_float(v.x)),
                  max_nan(__uint_as_float(v.y), max_nan(__uint_as_float(v.z), __uint_as_float(v.w))));
  }
  __device__ static __forceinline__ float max_finish(const MaxAcc& s) { return s.a; }
  __device__ static __forceinline__ void mass_vec(const uint4& v, u64 m2, u64 c2, u64& acc) {
    acc = add2(acc, mass2(pk2(v.x, v.y), m2, c2));
    acc = add2(acc, mass2(pk2(v.z, v.w), m2, c2));
  }
  __device__ static __forceinline__ uint32_t thr_pack(uint32_t bits) { return bits; }
  __device__ static __forceinline__ bool any_ge(const uint4& v, uint32_t thr) {
    const float t = __uint_as_float(thr);
    return (__uint_as_float(v.x) >= t) | (__uint_as_float(v.y) >= t) | (__uint_as_float(v.z) >= t) |
           (__uint_as_float(v.w) >= t);
  }
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
  __device__ static __forceinline__ bool any_eq(const uint4& v, uint32_t thr) { return mask_eq(v, thr) != 0u; }
};

// ------------------------------------------------------------ row state

struct RowStat {
  float m;               // row maximum
  uint32_t kmax;         // key of m
  uint32_t kstar;        // kept iff key > kstar, or key == kstar and (not partial or index < tie_cut)
  uint32_t cstar;        // kept tokens of value kstar: the lowest-index ones
  uint32_t tie_total;    // tokens of value kstar in the row
  int tie_cut;           // partial rows: index of the first kstar-valued token that is not kept
  uint32_t thr;          // packed value of kstar (quick skips, equality tests)
  double zkept;          // sum of masses over the kept set
  float inv_z;
  int all_kept;
  int bad;
  int partial;           // cstar < tie_total
};

struct Shm {
  // exchange slots, read by the other CTAs of the cluster
  float x_max[2];
  double x_sum[2];
  uint32_t x_tie[2];
  double x_res[2];
  double x_pm[2];
  uint32_t x_pc[2];
  uint32_t x_pk[2];
  // CTA scratch
  float w_max[kWarps][2];
  float w_sum[kWarps][2];
  float w_res[kWarps];
  uint32_t w_u[kWarps];
  float w_f[kWarps];
  uint32_t w_tie[kWarps][2];
  double w_pm[kWarps];
  uint32_t w_pc[kWarps];
  uint32_t w_pk[kWarps];
  double b_zfull[2];
  double b_S, b_Pc;
  int b_owner;
  uint32_t b_dlb[2];
  int c_found;
  uint32_t c_d, c_c, c_t;
  double c_z;
  uint32_t tie_before[2], tie_local[2];
  uint32_t pc[2][kBinThreads];  // per-thread count of its four histogram bins
  float pm[2][kBinThreads];     // per-thread mass of its four histogram bins
  int tie_cut[2];
  int tie_warp[2];
  uint32_t tie_j[2];
  uint32_t fb_need[2];
  int draw_warp;
  double draw_base;
  RowStat rs[2];
  alignas(8) uint64_t mbar;
};

template <int DT>
__device__ __forceinline__ float value_of_key(uint32_t k) {
  return Elt<DT>::value(Elt<DT>::bits_of_key(k));
}

// Fixed-order sum of one double per cluster rank (lane c holds rank c's).
template <int CS>
__device__ __forceinline__ double cluster_sum_f64(double mine_lane_c) {
  double z = 0.0;
#pragma unroll
  for (int c = 0; c < CS; ++c) z += __shfl_sync(kFull, mine_lane_c, c);
  return z;
}

// One element of a shared-memory row buffer.
template <int DT>
__device__ __forceinline__ uint32_t lds_elem(uint32_t base, int t) {
  return DT == DT_BF16 ? lds_u16(base + 2u * static_cast<uint32_t>(t)) : lds_u32(base + 4u * static_cast<uint32_t>(t));
}

// Kept test for the element of index t (whole-row index) with the given key.
__device__ __forceinline__ bool kept_key(const RowStat& rs, uint32_t key, int t) {
  if (rs.all_kept) return true;
  if (key > rs.kstar) return true;
  return key == rs.kstar && (!rs.partial || t < rs.tie_cut);
}

// Bit j set for the elements of vector v (CTA-local) that lie inside the slice.
template <int DT>
__device__ __forceinline__ uint32_t valid_mask(int v, int n) {
  const int left = n - v * Elt<DT>::kPerVec;
  return left >= Elt<DT>::kPerVec ? (1u << Elt<DT>::kPerVec) - 1u : (left > 0 ? (1u << left) - 1u : 0u);
}

// Draw weights of the elements of one 16-byte vector: w = max(0, p - q)
// (residual) or w = p (bonus).  t0 is the vector's first CTA-local element,
// lo the slice start.  Vectors with no element at or above the target's cut
// value are skipped with one packed compare.
template <int DT>
__device__ __forceinline__ float vec_weights(const uint4& xp, const uint4& xq, int t0, int lo, int n, bool use_q,
                                             const RowStat& rp, const RowStat& rq, float cexp, float* w) {
  using E = Elt<DT>;
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < E::kPerVec; ++j) w[j] = 0.f;
  if (!rp.all_kept && !Hot<DT>::any_ge(xp, rp.thr)) return 0.f;
#pragma unroll
  for (int j = 0; j < E::kPerVec; ++j) {
    if (t0 + j < n) {
      const int t = lo + t0 + j;
      const uint32_t bp = E::bits_of(xp, j);
      float pv = 0.f;
      if (kept_key(rp, E::key(bp), t)) pv = softmax_mass(E::value(bp), rp.m, cexp) * rp.inv_z;
      if (use_q) {
        const uint32_t bq = E::bits_of(xq, j);
        float qv = 0.f;
        if (kept_key(rq, E::key(bq), t)) qv = softmax_mass(E::value(bq), rq.m, cexp) * rq.inv_z;
        w[j] = fmaxf(pv - qv, 0.f);
      } else {
        w[j] = pv;
      }
      s += w[j];
    }
  }
  return s;
}

// ------------------------------------------------------ CTA-wide scans

// Exclusive prefix (thread order) of a u32 over the CTA; `total` gets the sum.
__device__ __forceinline__ uint32_t block_excl_u32(uint32_t v, uint32_t* wtmp, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = warp_incl_scan_u32(v);
  if (lane == 31) wtmp[warp] = incl;
  __syncthreads();
  uint32_t off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t x = wtmp[w];
    if (w < warp) off += x;
    tot += x;
  }
  __syncthreads();
  total = tot;
  return off + incl - v;
}

// Exclusive prefix (thread order) of a float over the CTA, as a double-float.
__device__ __forceinline__ DF block_excl_f32(float v, float* wtmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float incl = warp_incl_scan(v);
  if (lane == 31) wtmp[warp] = incl;
  __syncthreads();
  DF off{0.f, 0.f};
  for (int w = 0; w < warp; ++w) off = df_add(off, wtmp[w]);
  __syncthreads();
  return df_add(off, incl - v);
}

// Smallest thread index whose flag is set, or -1.
__device__ __forceinline__ int block_first(bool f, uint32_t* wtmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned ball = __ballot_sync(kFull, f);
  if (lane == 0) wtmp[warp] = ball ? static_cast<uint32_t>(warp * 32 + __ffs(ball) - 1) : 0xFFFFFFFFu;
  __syncthreads();
  uint32_t first = 0xFFFFFFFFu;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) first = min(first, wtmp[w]);
  __syncthreads();
  return first == 0xFFFFFFFFu ? -1 : static_cast<int>(first);
}

// Sum over the cluster of bins 4t .. 4t+3 of one row's histogram (hrow: the
// shared-window address of this CTA's copy).
template <int CS>
__device__ __forceinline__ uint4 cluster_bins4(uint32_t hrow, int t) {
  uint4 part[CS];
#pragma unroll
  for (int c = 0; c < CS; ++c) part[c] = ld_cluster_v4(mapa_shared(hrow + 16u * static_cast<uint32_t>(t), c));
  uint4 s = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int c = 0; c < CS; ++c) {
    s.x += part[c].x;
    s.y += part[c].y;
    s.z += part[c].z;
    s.w += part[c].w;
  }
  return s;
}

__device__ __forceinline__ uint32_t u4_at(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Stage 1 of the cut (all threads): thread t publishes the cluster-wide count
// and mass of its four bins 4t .. 4t+3 (bin d: tokens of value key kmax - d).
template <int DT, int CS>
__device__ __forceinline__ void bins_partials(Shm& sh, int r, uint32_t hrow, int nbins, uint32_t kmax, float m,
                                              float cexp) {
  const int t = threadIdx.x;
  if (t >= kBinThreads) return;
  uint32_t C = 0u;
  float M = 0.f;
  if (4 * t < nbins) {
    const uint4 b = cluster_bins4<CS>(hrow, t);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int d = 4 * t + i;
      const uint32_t c = d < nbins ? u4_at(b, i) : 0u;
      if (c) {
        C += c;
        M += static_cast<float>(c) * softmax_mass(value_of_key<DT>(kmax - static_cast<uint32_t>(d)), m, cexp);
      }
    }
  }
  sh.pc[r][t] = C;
  sh.pm[r][t] = M;
}

// Stage 2 of the cut (one warp per row).  Top-k: the bin where the running
// count reaches top_k (exact, integer); its tokens kept are the
// top_k - (count before) lowest-index ones.  Top-p (on the top-k set if
// any): the first bin where the running mass reaches top_p * Z_k; a token of
// that value is kept while the mass ranked before it stays below the
// target.  Lane l scans bin threads 4l .. 4l+3; the thread holding the crossing
// re-reads its four bins.  Returns false if the cut lies beyond the counted
// bins (the exact fallback then takes over).
template <int DT, int CS>
__device__ __noinline__ bool cut_scan_warp(Shm& sh, int r, uint32_t hrow, int nbins, RowStat& rs, int top_k, float top_p,
                              double zfull, float cexp) {
  const int lane = threadIdx.x & 31;
  const bool topk_on = top_k > 0, topp_on = top_p < 1.f;
  const uint32_t K = static_cast<uint32_t>(top_k);
  uint32_t dk = 0xFFFFFFFFu, ck = 0u, tk = 0u;
  int tkthr = kThreads;  // thread holding the top-k bin
  double zk = zfull;
  if (topk_on) {
    constexpr int kL = kBinThreads / 32;  // bin threads per lane
    uint32_t lc[kL], C = 0u;
    DF M{0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kL; ++i) {
      lc[i] = sh.pc[r][kL * lane + i];
      C += lc[i];
      M = df_add(M, sh.pm[r][kL * lane + i]);
    }
    const uint32_t incl = warp_incl_scan_u32(C);
    const DF Mi = warp_incl_scan_df(M);
    const unsigned ball = __ballot_sync(kFull, incl - C < K && incl >= K);
    if (!ball) return false;
    const int L = __ffs(ball) - 1;
    uint32_t o_d = 0u, o_c = 0u, o_t = 0u;
    int o_thr = 0;
    double o_z = 0.0;
    if (lane == L) {
      uint32_t run = incl - C;
      DF mrun = df_add(Mi, -M.hi);
      mrun = df_add(mrun, -M.lo);
      int t = kL * L;
#pragma unroll
      for (int i = 0; i < kL; ++i) {
        if (run + lc[i] >= K) { t = kL * L + i; break; }
        run += lc[i];
        mrun = df_add(mrun, sh.pm[r][kL * L + i]);
      }
      const uint4 b = cluster_bins4<CS>(hrow, t);
      for (int j = 0; j < 4; ++j) {
        const int d = 4 * t + j;
        const uint32_t c = d < nbins ? u4_at(b, j) : 0u;
        const float e = c ? softmax_mass(value_of_key<DT>(rs.kmax - static_cast<uint32_t>(d)), rs.m, cexp) : 0.f;
        if (run + c >= K) {
          o_d = static_cast<uint32_t>(d);
          o_c = K - run;
          o_t = c;
          o_thr = t;
          o_z = df_value(mrun) + (double)(K - run) * (double)e;
          break;
        }
        run += c;
        mrun = df_add(mrun, static_cast<float>(c) * e);
      }
    }
    dk = __shfl_sync(kFull, o_d, L);
    ck = __shfl_sync(kFull, o_c, L);
    tk = __shfl_sync(kFull, o_t, L);
    tkthr = __shfl_sync(kFull, o_thr, L);
    zk = __shfl_sync(kFull, o_z, L);
  }
  uint32_t dstar = dk, cstar = ck, tstar = tk;
  double zkept = zk;
  if (topp_on) {
    const DF tdf = df_from((double)top_p * zk);
    // lane masses over the top-k set: threads past the top-k bin hold nothing,
    // the thread holding it only its bins up to dk (with ck tokens at dk)
    constexpr int kL = kBinThreads / 32;
    DF M{0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kL; ++i) {
      const int t = kL * lane + i;
      if (t < tkthr) M = df_add(M, sh.pm[r][t]);
    }
    if (topk_on && tkthr / kL == lane) {
      const uint4 b = cluster_bins4<CS>(hrow, tkthr);
      for (int j = 0; j < 4; ++j) {
        const uint32_t d = static_cast<uint32_t>(4 * tkthr + j);
        if (d > dk) break;
        const uint32_t c = d == dk ? ck : u4_at(b, j);
        if (c) M = df_add(M, static_cast<float>(c) * softmax_mass(value_of_key<DT>(rs.kmax - d), rs.m, cexp));
      }
    }
    const DF Mi = warp_incl_scan_df(M);
    const unsigned ball = __ballot_sync(kFull, (M.hi > 0.f) && df_diff(Mi, tdf) >= 0.f);
    if (!ball) return false;
    const int L = __ffs(ball) - 1;
    uint32_t o_d = 0u, o_c = 0u, o_t = 0u;
    double o_z = 0.0;
    int found = 0;
    if (lane == L) {
      const double target = df_value(tdf);
      double run = df_value(Mi) - df_value(M);  // mass of the lanes before
      int tlast = -1;
      double runlast = run;
      for (int i = 0; i < kL && !found; ++i) {
        const int t = kL * L + i;
        if (t > tkthr) break;
        const uint4 b = cluster_bins4<CS>(hrow, t);
        for (int j = 0; j < 4; ++j) {
          const uint32_t d = static_cast<uint32_t>(4 * t + j);
          if (static_cast<int>(d) >= nbins || (topk_on && d > dk)) break;
          uint32_t c = u4_at(b, j);
          const uint32_t real = c;
          if (topk_on && d == dk) c = ck;
          if (!c) continue;
          const float e = softmax_mass(value_of_key<DT>(rs.kmax - d), rs.m, cexp);
          const double me = (double)c * (double)e;
          tlast = static_cast<int>(d);
          runlast = run;
          if (run + me >= target) {
            const float xneed = static_cast<float>((target - run) / (double)e);
            uint32_t cp = c;
            if (xneed < static_cast<float>(c)) cp = max(1u, static_cast<uint32_t>(ceilf(xneed)));
            o_d = d;
            o_c = cp;
            o_t = real;
            o_z = run + (double)cp * (double)e;
            found = 1;
            break;
          }
          run += me;
        }
      }
      if (!found && tlast >= 0) {  // rounding: the last non-empty bin takes the cut
        const uint32_t d = static_cast<uint32_t>(tlast);
        const uint4 b = cluster_bins4<CS>(hrow, tlast / 4);
        uint32_t c = u4_at(b, tlast % 4);
        o_t = c;
        if (topk_on && d == dk) c = ck;
        const float e = softmax_mass(value_of_key<DT>(rs.kmax - d), rs.m, cexp);
        o_d = d;
        o_c = c;
        o_z = runlast + (double)c * (double)e;
        found = 1;
      }
    }
    if (!__shfl_sync(kFull, found, L)) return false;
    dstar = __shfl_sync(kFull, o_d, L);
    cstar = __shfl_sync(kFull, o_c, L);
    tstar = __shfl_sync(kFull, o_t, L);
    zkept = __shfl_sync(kFull, o_z, L);
  }
  rs.kstar = rs.kmax - dstar;
  rs.cstar = cstar;
  rs.tie_total = tstar;
  rs.zkept = zkept;
  rs.partial = cstar < tstar ? 1 : 0;
  return true;
}

// Smallest d such that bins 0..d of a CTA-local histogram hold >= need
// tokens; kWindow - 1 if they never do.  All threads call it.
__device__ __noinline__ uint32_t local_bins_reach(uint32_t hrow, uint32_t need, Shm& sh) {
  constexpr int kB = 4;
  const int tid = threadIdx.x;
  const uint4 b4 = tid < kBinThreads ? lds128(hrow + 16u * tid) : make_uint4(0u, 0u, 0u, 0u);
  const uint32_t cnt[kB] = {b4.x, b4.y, b4.z, b4.w};
  uint32_t C = cnt[0] + cnt[1] + cnt[2] + cnt[3];
  uint32_t total;
  const uint32_t P = block_excl_u32(C, sh.w_u, total);
  if (tid == 0) sh.c_d = static_cast<uint32_t>(kWindow - 1);
  __syncthreads();
  if (P < need && P + C >= need) {
    uint32_t run = P;
#pragma unroll
    for (int i = 0; i < kB; ++i) {
      if (run < need && run + cnt[i] >= need) sh.c_d = static_cast<uint32_t>(tid * kB + i);
      run += cnt[i];
    }
  }
  __syncthreads();
  const uint32_t d = sh.c_d;
  __syncthreads();
  return d;
}

enum PassKind { PASS_COUNT_GE = 0, PASS_MASS_GT = 1, PASS_MIN_GE = 2, PASS_COUNT_EQ = 3 };

// One full pass over this CTA's slice of one row, reduced over the cluster.
// Used only by the exact fallback search of the cut.
template <int DT, int CS>
__device__ __noinline__ double cluster_pass(cg::cluster_group& cluster, Shm& sh, uint32_t buf, int n, int nvec, int kind,
                               uint32_t kappa, float m, float c, uint32_t& slot) {
  using E = Elt<DT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t cnt = 0, kmin = 0xFFFFFFFFu;
  float mass = 0.f;
  for (int v = tid; v < nvec; v += kThreads) {
    const uint4 x = lds128(buf + 16u * v);
    const int t0 = v * E::kPerVec;
#pragma unroll
    for (int j = 0; j < E::kPerVec; ++j) {
      if (t0 + j < n) {
        const uint32_t b = E::bits_of(x, j);
        const uint32_t k = E::key(b);
        if (kind == PASS_COUNT_GE) cnt += (k >= kappa);
        else if (kind == PASS_COUNT_EQ) cnt += (k == kappa);
        else if (kind == PASS_MIN_GE) { if (k >= kappa) kmin = min(kmin, k); }
        else if (k > kappa) mass += softmax_mass(E::value(b), m, c);
      }
    }
  }
  const uint32_t s = slot & 1u;
  mass = warp_sum_f32(mass);
  cnt = warp_sum_u32(cnt);
  kmin = warp_min_u32(kmin);
  if (lane == 0) { sh.w_pm[warp] = mass; sh.w_pc[warp] = cnt; sh.w_pk[warp] = kmin; }
  __syncthreads();
  if (tid == 0) {
    double tm = 0.0;
    uint32_t tc = 0, tk = 0xFFFFFFFFu;
    for (int w = 0; w < kWarps; ++w) { tm += sh.w_pm[w]; tc += sh.w_pc[w]; tk = min(tk, sh.w_pk[w]); }
    sh.x_pm[s] = tm; sh.x_pc[s] = tc; sh.x_pk[s] = tk;
  }
  cluster.sync();
  double res;
  {
    double vm = 0.0;
    uint32_t vc = 0, vk = 0xFFFFFFFFu;
    if (lane < CS) {
      const Shm* peer = cluster.map_shared_rank(&sh, lane);
      vm = peer->x_pm[s]; vc = peer->x_pc[s]; vk = peer->x_pk[s];
    }
    if (kind == PASS_MASS_GT) res = cluster_sum_f64<CS>(vm);
    else if (kind == PASS_MIN_GE) res = (double)warp_min_u32(vk);
    else res = (double)warp_sum_u32(vc);
  }
  ++slot;
  return res;
}

// Largest bf16 / fp32 value not above v (v finite), as bits.
template <int DT>
__device__ __forceinline__ uint32_t bits_round_down(float v) {
  const uint32_t u = __float_as_uint(v);
  if (DT == DT_F32) return u;
  const uint32_t hi = u >> 16;
  if ((u & 0xFFFFu) == 0u) return hi;
  return (u & 0x80000000u) ? hi + 1u : hi;  // negative: away from zero is down
}

// The exact cut of one row by a bitwise search over the keys: used when the
// cut lies outside the exact-value histogram (flat rows, fp32 rows).  Every
// step is a full pass over the slice reduced over the cluster.
template <int DT, int CS>
__device__ __noinline__ void fallback_row(cg::cluster_group& cluster, Shm& sh, uint32_t bb, int n, int nvec, int r,
                                          int top_k, float top_p, double zfull_r, float cexp, uint32_t& slot) {
  using E = Elt<DT>;
  using H = Hot<DT>;
  const int tid = threadIdx.x;
  const bool topk_on = top_k > 0, topp_on = top_p < 1.f;
  RowStat rs = sh.rs[r];
  const int kb = E::kKeyBits;
  uint32_t kk = 0, ck = 0, tk = 0;
  double zk = zfull_r;
  if (topk_on) {
    for (int bit = kb - 1; bit >= 0; --bit) {
      const uint32_t cand = kk | (1u << bit);
      const double cnt = cluster_pass<DT, CS>(cluster, sh, bb, n, nvec, PASS_COUNT_GE, cand, rs.m, cexp, slot);
      if (cnt >= (double)top_k) kk = cand;
    }
    const uint32_t gt = (kk == 0xFFFFFFFFu) ? 0u
        : static_cast<uint32_t>(cluster_pass<DT, CS>(cluster, sh, bb, n, nvec, PASS_COUNT_GE, kk + 1u, rs.m, cexp, slot));
    ck = static_cast<uint32_t>(top_k) - gt;
    tk = static_cast<uint32_t>(cluster_pass<DT, CS>(cluster, sh, bb, n, nvec, PASS_COUNT_EQ, kk, rs.m, cexp, slot));
    const float ek = softmax_mass(value_of_key<DT>(kk), rs.m, cexp);
    zk = cluster_pass<DT, CS>(cluster, sh, bb, n, nvec, PASS_MASS_GT, kk, rs.m, cexp, slot) + (double)ck * (double)ek;
  }
  uint32_t kstar = kk, cstar = ck, tstar = tk;
  double zkept = zk;
  if (topp_on) {
    const double target = (double)top_p * zk;
    // G(kappa): mass of the top-k set strictly above kappa
    auto G = [&](uint32_t kappa) -> double {
      if (topk_on && kappa < kk) return zk;
      return cluster_pass<DT, CS>(cluster, sh, bb, n, nvec, PASS_MASS_GT, kappa, rs.m, cexp, slot);
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
    kstar = static_cast<uint32_t>(cluster_pass<DT, CS>(cluster, sh, bb, n, nvec, PASS_MIN_GE, k0, rs.m, cexp, slot));
    const double mb = G(kstar);
    tstar = static_cast<uint32_t>(cluster_pass<DT, CS>(cluster, sh, bb, n, nvec, PASS_COUNT_EQ, kstar, rs.m, cexp, slot));
    const uint32_t avail = (topk_on && kstar == kk) ? ck : tstar;
    const float ep = softmax_mass(value_of_key<DT>(kstar), rs.m, cexp);
    const double xneed = (target - mb) / (double)ep;
    uint32_t cp = avail;
    if (xneed < (double)avail) cp = max(1u, static_cast<uint32_t>(ceil(xneed)));
    cstar = cp;
    zkept = mb + (double)cp * (double)ep;
  }
  rs.kstar = kstar;
  rs.cstar = cstar;
  rs.tie_total = tstar;
  rs.zkept = zkept;
  rs.partial = cstar < tstar ? 1 : 0;
  rs.inv_z = 1.f / static_cast<float>(zkept);
  rs.thr = H::thr_pack(E::bits_of_key(kstar));
  __syncthreads();
  if (tid == 0) sh.rs[r] = rs;
  __syncthreads();
}

// Where a partial tie stops.  The kept tokens of value kstar are the cstar
// lowest-index ones.  Each CTA needs the number of such tokens in lower
// cluster ranks (from the exchanged histograms, or, for rows cut by the
// fallback search, from one more exchange); the CTA holding the first one not
// kept finds its index, every other CTA records a bound outside its slice.
template <int DT, int CS, int NR>
__device__ __noinline__ void tie_cuts(cg::cluster_group& cluster, Shm& sh, uint32_t buf0, uint32_t buf1,
                                      uint32_t hist, int lo, int hi, int n, int V, bool part_fb) {
  using E = Elt<DT>;
  using H = Hot<DT>;
  const int crank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = (n * E::kBytes + 15) / 16;
  const int vpw = ((nvec + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int seg_beg = min(nvec, warp * vpw);
  const int seg_end = min(nvec, seg_beg + vpw);
  const int seg_iters = (seg_end - seg_beg + 31) / 32;
  const uint32_t buf[2] = {buf0, buf1};
  if (warp < NR && sh.rs[warp].partial && !sh.fb_need[warp]) {
    const int r = warp;
    const uint32_t dstar = sh.rs[r].kmax - sh.rs[r].kstar;
    uint32_t v = 0u;
    if (lane < CS) v = ld_cluster_u32(mapa_shared(hist + 4u * (r * kWindow + dstar), lane));
    const uint32_t before = warp_sum_u32(lane < crank ? v : 0u);
    const uint32_t local = __shfl_sync(kFull, v, crank);
    if (lane == 0) { sh.tie_before[r] = before; sh.tie_local[r] = local; }
  }
  if (part_fb) {  // rows cut by the fallback: count per CTA, then exchange
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      uint32_t c = 0;
      if (sh.rs[r].partial && sh.fb_need[r]) {
        const uint32_t thr = sh.rs[r].thr;
        for (int v = seg_beg + lane; v < seg_end; v += 32)
          c += __popc(H::mask_eq(lds128(buf[r] + 16u * v), thr) & valid_mask<DT>(v, n));
      }
      c = warp_sum_u32(c);
      if (lane == 0) sh.w_tie[warp][r] = c;
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        uint32_t t = 0;
        for (int w = 0; w < kWarps; ++w) t += sh.w_tie[w][r];
        sh.x_tie[r] = t;
      }
    }
    cluster.sync();  // ------------------------------------- sync: fallback ties
    if (warp < NR && sh.rs[warp].partial && sh.fb_need[warp]) {
      const int r = warp;
      uint32_t v = 0u;
      if (lane < CS) v = cluster.map_shared_rank(&sh, lane)->x_tie[r];
      const uint32_t before = warp_sum_u32(lane < crank ? v : 0u);
      if (lane == 0) { sh.tie_before[r] = before; sh.tie_local[r] = sh.x_tie[r]; }
    }
  }
  __syncthreads();
  bool search = false;
  if (tid == 0) {
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      sh.tie_warp[r] = -1;
      sh.tie_cut[r] = V;
      if (!sh.rs[r].partial) continue;
      const int64_t j = static_cast<int64_t>(sh.rs[r].cstar) - sh.tie_before[r];
      if (j <= 0) sh.tie_cut[r] = lo;
      else if (j >= static_cast<int64_t>(sh.tie_local[r])) sh.tie_cut[r] = hi;
      else { sh.tie_cut[r] = -1; sh.tie_j[r] = static_cast<uint32_t>(j); }
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < NR; ++r) search |= sh.tie_cut[r] < 0;
  if (search) {  // this CTA holds the first tie token that is not kept
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      uint32_t c = 0;
      if (sh.tie_cut[r] < 0) {
        const uint32_t thr = sh.rs[r].thr;
        for (int v = seg_beg + lane; v < seg_end; v += 32)
          c += __popc(H::mask_eq(lds128(buf[r] + 16u * v), thr) & valid_mask<DT>(v, n));
      }
      c = warp_sum_u32(c);
      if (lane == 0) sh.w_tie[warp][r] = c;
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (sh.tie_cut[r] >= 0) continue;
        uint32_t run = 0;
        for (int w = 0; w < kWarps; ++w) {
          if (run + sh.w_tie[w][r] > sh.tie_j[r]) {
            sh.tie_warp[r] = w;
            sh.tie_j[r] -= run;
            break;
          }
          run += sh.w_tie[w][r];
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      if (warp != sh.tie_warp[r]) continue;
      const uint32_t thr = sh.rs[r].thr;
      uint32_t jj = sh.tie_j[r];
      for (int it = 0; it < seg_iters; ++it) {
        const int v = seg_beg + it * 32 + lane;
        const uint32_t msk = v < seg_end ? (H::mask_eq(lds128(buf[r] + 16u * v), thr) & valid_mask<DT>(v, n)) : 0u;
        const uint32_t c = __popc(msk);
        const uint32_t incl = warp_incl_scan_u32(c);
        const uint32_t tot = __shfl_sync(kFull, incl, 31);
        if (jj < tot) {
          if (incl > jj && incl - c <= jj) {  // this lane holds the token
            uint32_t mm = msk;
            for (uint32_t q = jj - (incl - c); q > 0; --q) mm &= mm - 1u;
            sh.tie_cut[r] = lo + v * E::kPerVec + (__ffs(mm) - 1);
          }
          break;
        }
        jj -= tot;
      }
    }
    __syncthreads();
  }
  if (tid == 0) {
#pragma unroll
    for (int r = 0; r < NR; ++r) sh.rs[r].tie_cut = sh.tie_cut[r];
  }
  __syncthreads();
}

// The filtered, normalised probabilities of this CTA's slice, written out.
template <int DT>
__device__ __noinline__ void write_probs(const SampleArgs& a, uint32_t buf0, const RowStat& rp, float cexp, int unit,
                                         int lo, int n, int V) {
  using E = Elt<DT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = (n * E::kBytes + 15) / 16;
  const int vpw = ((nvec + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int seg_beg = min(nvec, warp * vpw);
  const int seg_end = min(nvec, seg_beg + vpw);
  const uint32_t buf[1] = {buf0};
  float* out = a.out_probs + static_cast<size_t>(unit) * V + lo;
  const bool vec_out = ((reinterpret_cast<uintptr_t>(out) & 15u) == 0) && (V % 4 == 0);
  for (int v = seg_beg + lane; v < seg_end; v += 32) {
    const int t0 = v * E::kPerVec;
    const uint4 x = lds128(buf[0] + 16u * v);
    float w[8];
    vec_weights<DT>(x, x, t0, lo, n, false, rp, rp, cexp, w);
    if (rp.bad) {
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = 0.f;
    }
    if (vec_out && t0 + E::kPerVec <= n) {
      reinterpret_cast<float4*>(out + t0)[0] = make_float4(w[0], w[1], w[2], w[3]);
      if (E::kPerVec == 8) reinterpret_cast<float4*>(out + t0)[1] = make_float4(w[4], w[5], w[6], w[7]);
    } else {
#pragma unroll
      for (int j = 0; j < E::kPerVec; ++j)
        if (t0 + j < n) out[t0 + j] = w[j];
    }
  }
}

// The CTA holding the drawn token finds it: the warp whose segment holds the
// crossing walks it vector by vector (index order) and writes the token.
template <int DT, int NR>
__device__ __noinline__ void draw_walk(const SampleArgs& a, Shm& sh, uint32_t buf0, uint32_t bufq, bool use_q,
                                       const RowStat& rp, const RowStat& rq, float cexp, double target, int lo,
                                       int n, int unit, int b) {
  using E = Elt<DT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = (n * E::kBytes + 15) / 16;
  const int vpw = ((nvec + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int seg_beg = min(nvec, warp * vpw);
  const int seg_end = min(nvec, seg_beg + vpw);
  const int seg_iters = (seg_end - seg_beg + 31) / 32;
  const int kq = a.k;
  const uint32_t buf[2] = {buf0, bufq};
  if (tid == 0) {
    double run = 0.0, wbase = 0.0, lbase = 0.0;
    int wsel = -1, wlast = -1;
    for (int w = 0; w < kWarps; ++w) {
      const double sw = (double)sh.w_res[w];
      if (sw > 0.0) { wlast = w; lbase = run; }
      if (wsel < 0 && sw > 0.0 && run + sw > target) { wsel = w; wbase = run; }
      run += sw;
    }
    if (wsel < 0) { wsel = wlast; wbase = lbase; }
    sh.draw_warp = wsel;
    sh.draw_base = wbase;
  }
  __syncthreads();
  if (warp == sh.draw_warp) {
    const float tw = static_cast<float>(target - sh.draw_base);
    float run = 0.f;
    int token = -1, last_pos = -1;
    for (int it = 0; it < seg_iters && token < 0; ++it) {
      const int v = seg_beg + it * 32 + lane;
      const bool valid = v < seg_end;
      const int t0 = v * E::kPerVec;
      float w[8];
      float ls = 0.f;
      int lpos = -1;
      if (valid) {
        const uint4 xp = lds128(buf[0] + 16u * v);
        const uint4 xq = use_q ? lds128(buf[NR - 1] + 16u * v) : xp;
        ls = vec_weights<DT>(xp, xq, t0, lo, n, use_q, rp, rq, cexp, w);
#pragma unroll
        for (int j = 0; j < E::kPerVec; ++j)
          if (w[j] > 0.f) lpos = t0 + j;
      }
      const float incl = warp_incl_scan(ls);
      const unsigned ball = __ballot_sync(kFull, valid && ls > 0.f && run + incl > tw);
      const int lastl = 31 - __clz(__ballot_sync(kFull, lpos >= 0) | 1u);
      const int lp = __shfl_sync(kFull, lpos, lastl);
      if (lp >= 0) last_pos = lp;
      if (ball) {
        const int l = __ffs(ball) - 1;
        int tok = -1;
        if (lane == l) {
          float cum = run + (incl - ls);
          int lastj = -1;
#pragma unroll
          for (int j = 0; j < E::kPerVec; ++j) {
            if (w[j] > 0.f) lastj = t0 + j;
            cum += w[j];
            if (tok < 0 && w[j] > 0.f && cum > tw) tok = t0 + j;
          }
          if (tok < 0) tok = lastj;
        }
        token = __shfl_sync(kFull, tok, l);
      }
      run += __shfl_sync(kFull, incl, 31);
    }
    if (token < 0) token = last_pos;  // only reachable through rounding
    if (lane == 0) {
      a.recs[unit].drawn = token >= 0 ? lo + token : -1;
      __threadfence();
      if (atomicAdd(a.tickets + b, 1u) == static_cast<uint32_t>(2 * kq)) sample_finalize(a, b);
    }
  }
}

// Bound for a top-p cut from the cluster's warp maxima (one warp per row).
// Those maxima are tokens of the row.  If the ones at or above a value v
// already weigh top_p * Z, the nucleus ends at or above v, so no token below v
// is kept.  (1e-4 of margin covers rounding.)  Writes the bound value (or
// -inf) to sh.w_f[r].
template <int CS>
__device__ __noinline__ void warp_max_bound(Shm& sh, int r, float m_r, double z_r, float cexp, float top_p) {
  const int lane = threadIdx.x & 31;
  constexpr int nw = kWarps * CS;
  float v0 = -INFINITY, v1 = -INFINITY;
  if (lane < nw) v0 = ld_cluster_f32(mapa_shared(smem_addr(&sh.w_max[lane % kWarps][r]), lane / kWarps));
  if (lane + 32 < nw)
    v1 = ld_cluster_f32(mapa_shared(smem_addr(&sh.w_max[(lane + 32) % kWarps][r]), (lane + 32) / kWarps));
  const float e0 = v0 > -INFINITY ? softmax_mass(v0, m_r, cexp) : 0.f;
  const float e1 = v1 > -INFINITY ? softmax_mass(v1, m_r, cexp) : 0.f;
  float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
  for (int j = 0; j < nw; ++j) {
    const float vj = __shfl_sync(kFull, j < 32 ? v0 : v1, j & 31);
    const float ej = __shfl_sync(kFull, j < 32 ? e0 : e1, j & 31);
    s0 += vj >= v0 ? ej : 0.f;
    s1 += vj >= v1 ? ej : 0.f;
  }
  const float target = 1.0001f * top_p * static_cast<float>(z_r);
  float cand = -INFINITY;
  if (v0 > -INFINITY && s0 >= target) cand = v0;
  if (v1 > -INFINITY && s1 >= target) cand = fmaxf(cand, v1);
  cand = warp_max(cand);
  if (lane == 0) sh.w_f[r] = cand;
}

}  // namespace

// One unit (b, pos) with NR rows (2: target and draft, 1: target only).
template <int DT, int CS, int NR>
__device__ __forceinline__ void unit_body(const SampleArgs& a, cg::cluster_group& cluster, Shm& sh,
                                          unsigned char* dsm, int unit, int b, int pos,
                                          const unsigned char* rowp, const unsigned char* rowq) {
  using E = Elt<DT>;
  using H = Hot<DT>;
  const int crank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;
  const float T = a.temperature_per_seq ? a.temperature_per_seq[b] : a.temperature;
  const bool bad_t = !(T > 0.f) || isinf(T);
  const float cexp = kLog2e / T;
  const u64 c2 = pkf(cexp, cexp);

  const int lo = min(V, crank * a.chunk);
  const int hi = min(V, lo + a.chunk);
  const int n = hi - lo;
  const int nvec = (n * E::kBytes + 15) / 16;
  const int nfull = n / E::kPerVec;  // vectors without a ragged tail
  const int bufbytes = ((a.chunk * E::kBytes + 15) / 16) * 16;
  // shared-window addresses of the two row buffers and of the histograms
  const uint32_t sbase = smem_addr(dsm);
  const uint32_t buf[2] = {sbase, sbase + static_cast<uint32_t>(bufbytes)};
  const uint32_t hist = sbase + 2u * static_cast<uint32_t>(bufbytes);
  unsigned char* const bufp[2] = {dsm, dsm + bufbytes};
  const unsigned char* rows[2] = {rowp, rowq};
  const bool aligned[2] = {a.aligned_target != 0, a.aligned_draft != 0};

  const bool topk_on = a.top_k > 0;
  const bool topp_on = a.top_p < 1.f;
  const bool filt = topk_on || topp_on;

  // warp segment: consecutive vectors, index order (iteration, lane, element)
  const int vpw = ((nvec + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int seg_beg = min(nvec, warp * vpw);
  const int seg_end = min(nvec, seg_beg + vpw);
  const int seg_iters = (seg_end - seg_beg + 31) / 32;

  // ------------------------------------------------------ phase 0: load
  if (tid == 0) {
    mbar_init(&sh.mbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t tx = 0;
#pragma unroll
    for (int r = 0; r < NR; ++r)
      if (aligned[r] && n > 0) tx += static_cast<uint32_t>(n * E::kBytes);
    mbar_arrive_expect_tx(&sh.mbar, tx);
#pragma unroll
    for (int r = 0; r < NR; ++r)
      if (aligned[r] && n > 0)
        bulk_copy_g2s(bufp[r], rows[r] + static_cast<size_t>(lo) * E::kBytes, static_cast<uint32_t>(n * E::kBytes),
                      &sh.mbar);
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    if (!aligned[r]) {
      for (int t = tid; t < n; t += kThreads) {
        const uint32_t bits = E::bits_at(rows[r], static_cast<int64_t>(lo) + t);
        if (E::kBytes == 2) sts_u16(buf[r] + 2u * t, bits);
        else sts_u32(buf[r] + 4u * t, bits);
      }
    }
  }
  if (filt)
    for (int t = tid; t < NR * kWindow; t += kThreads) sts_u32(hist + 4u * t, 0u);
  if (tid == 0 && !mbar_wait_bounded(&sh.mbar, 0)) set_status(a.status, SPEC_STATUS_TIMEOUT);
  __syncthreads();

  // ------------------------------------------------------ phase 1: max
  float tmax[NR];  // this thread's own maximum, for the top-k bound below
  {
    typename H::MaxAcc st[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) H::max_init(st[r]);
    int v = tid;
    for (; v + kThreads < nfull; v += 2 * kThreads) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        H::max_vec(lds128(buf[r] + 16u * v), st[r]);
        H::max_vec(lds128(buf[r] + 16u * (v + kThreads)), st[r]);
      }
    }
    if (v < nfull) {
#pragma unroll
      for (int r = 0; r < NR; ++r) H::max_vec(lds128(buf[r] + 16u * v), st[r]);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      float mx = H::max_finish(st[r]);
      for (int t = nfull * E::kPerVec + tid; t < n; t += kThreads) mx = max_nan(mx, E::value(lds_elem<DT>(buf[r], t)));
      tmax[r] = mx;
      mx = warp_max_nan(mx);
      if (lane == 0) sh.w_max[warp][r] = mx;
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        float m = -INFINITY;
        for (int w = 0; w < kWarps; ++w) m = max_nan(m, sh.w_max[w][r]);
        sh.x_max[r] = m;
      }
    }
  }
  cluster.sync();  // ---------------------------------------------- sync: max
  float m[NR];
  bool rbad[NR];
  uint32_t kmax[NR];
  bool any_bad = bad_t;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float pm = -INFINITY;
    if (lane < CS) pm = cluster.map_shared_rank(&sh, lane)->x_max[r];
    m[r] = warp_max_nan(pm);
    rbad[r] = bad_t || !isfinite(m[r]);  // NaN, +inf, or no finite entry
    any_bad |= rbad[r];
    const uint32_t mbits = (E::kBytes == 2) ? (__float_as_uint(m[r]) >> 16) : __float_as_uint(m[r]);
    kmax[r] = E::key(mbits);
  }

  // --------------------------------------- phase 2: sum of masses (if used)
  const bool need_sum = !topk_on;
  double zfull[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) zfull[r] = 0.0;
  if (need_sum) {
    if (!any_bad) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const u64 m2 = pkf(m[r], m[r]);
        u64 acc0 = 0ull, acc1 = 0ull;
        int v = tid;
        for (; v + kThreads < nfull; v += 2 * kThreads) {
          H::mass_vec(lds128(buf[r] + 16u * v), m2, c2, acc0);
          H::mass_vec(lds128(buf[r] + 16u * (v + kThreads)), m2, c2, acc1);
        }
        if (v < nfull) H::mass_vec(lds128(buf[r] + 16u * v), m2, c2, acc0);
        float s0, s1, s2, s3;
        upk(acc0, s0, s1);
        upk(acc1, s2, s3);
        float s = (s0 + s1) + (s2 + s3);
        for (int t = nfull * E::kPerVec + tid; t < n; t += kThreads)
          s += softmax_mass(E::value(lds_elem<DT>(buf[r], t)), m[r], cexp);
        s = warp_sum_f32(s);
        if (lane == 0) sh.w_sum[warp][r] = s;
      }
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        double s = 0.0;
        if (!any_bad)
          for (int w = 0; w < kWarps; ++w) s += (double)sh.w_sum[w][r];
        sh.x_sum[r] = s;
      }
    }
    cluster.sync();  // -------------------------------------------- sync: sum
    if (tid == 0) {  // fixed-order cluster total, one thread, then broadcast
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        double z = 0.0;
        for (int c = 0; c < CS; ++c) z += cluster.map_shared_rank(&sh, c)->x_sum[r];
        sh.b_zfull[r] = z;
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < NR; ++r) zfull[r] = sh.b_zfull[r];
  }

  // ------------------------- phase 3: exact-value histogram near the top
  // Bins d = kmax - key count the tokens of one value each.  Only tokens that
  // can survive the cut are counted:
  //  - at most kWindow values below the maximum;
  //  - top-k: none below this CTA's top_k-th largest thread maximum (that
  //    value is at most the top_k-th largest token of the row);
  //  - top-p alone: no token whose mass is below (1 - top_p) Z / V (all
  //    tokens ranked at or below it weigh less than (1 - top_p) Z, so the
  //    mass ranked before it exceeds top_p Z); half of that bound is used,
  //    as margin for rounding.
  uint32_t klo[NR];
  if (filt) {
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      uint32_t kl = kmax[r] >= static_cast<uint32_t>(kWindow - 1) ? kmax[r] - static_cast<uint32_t>(kWindow - 1) : 0u;
      const uint32_t kninf = E::key(E::kBytes == 2 ? 0xFF80u : 0xFF800000u);  // -inf
      if (kl < kninf) kl = kninf;
      if (topp_on && !topk_on && !any_bad && zfull[r] > 0.0) {
        const float lim = 0.5f * (1.f - a.top_p) * static_cast<float>(zfull[r]) / static_cast<float>(V);
        const float vb = m[r] + log2f(lim) / cexp;
        if (isfinite(vb) && vb > -3.0e38f) {
          const uint32_t kb = E::key(bits_round_down<DT>(vb));
          if (kb > kl) kl = kb;
        }
      }
      klo[r] = kl;
    }
    if (topp_on && !topk_on && !any_bad) {
      // a tighter bound from the cluster's warp maxima
      if (warp < NR)
        warp_max_bound<CS>(sh, warp, warp == 0 ? m[0] : m[NR - 1], warp == 0 ? zfull[0] : zfull[NR - 1], cexp, a.top_p);
      __syncthreads();
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float cand = sh.w_f[r];
        if (cand > -INFINITY) {
          const uint32_t cb = (E::kBytes == 2) ? (__float_as_uint(cand) >> 16) : __float_as_uint(cand);
          const uint32_t kc = E::key(cb);
          if (kc > klo[r]) klo[r] = kc;
        }
      }
      __syncthreads();
    }
    if (topk_on && !any_bad && a.top_k <= kThreads) {
      // histogram of the thread maxima, then this CTA's top_k-th largest
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (tmax[r] > -INFINITY) {
          const uint32_t tb = (E::kBytes == 2) ? (__float_as_uint(tmax[r]) >> 16) : __float_as_uint(tmax[r]);
          const uint32_t d = kmax[r] - E::key(tb);
          if (d < static_cast<uint32_t>(kWindow)) red_add_shared(hist + 4u * (r * kWindow + d), 1u);
        }
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const uint32_t dlb = local_bins_reach(hist + 4u * r * kWindow, static_cast<uint32_t>(a.top_k), sh);
        if (kmax[r] - dlb > klo[r]) klo[r] = kmax[r] - dlb;
      }
      for (int t = tid; t < NR * kWindow; t += kThreads) sts_u32(hist + 4u * t, 0u);
      __syncthreads();
    }
    if (!any_bad) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const uint32_t thr = H::thr_pack(E::bits_of_key(klo[r]));
        const uint32_t hr = hist + 4u * r * kWindow;
        const uint32_t km = kmax[r];
        for (int v = tid; v < nfull; v += kThreads) {
          const uint4 x = lds128(buf[r] + 16u * v);
          if (!H::any_ge(x, thr)) continue;
          uint32_t msk = H::mask_ge(x, thr);
          while (msk) {
            const int j = __ffs(msk) - 1;
            msk &= msk - 1u;
            red_add_shared(hr + 4u * (km - E::key(E::bits_of(x, j))), 1u);
          }
        }
        for (int t = nfull * E::kPerVec + tid; t < n; t += kThreads) {
          const uint32_t k = E::key(lds_elem<DT>(buf[r], t));
          if (k >= klo[r]) red_add_shared(hr + 4u * (km - k), 1u);
        }
      }
    }
    __syncthreads();
    cluster.sync();  // ---------------------------------------- sync: histogram
  }

  // ------------------------------------ phase 3b: the kept set of each row
  if (filt && !any_bad) {
#pragma unroll
    for (int r = 0; r < NR; ++r)
      bins_partials<DT, CS>(sh, r, hist + 4u * r * kWindow, static_cast<int>(kmax[r] - klo[r]) + 1, kmax[r], m[r],
                            cexp);
    __syncthreads();
  }
  if (warp < NR) {
    const int r = warp;
    // this warp's row, picked without a run-time array index
    const float m_r = r == 0 ? m[0] : m[NR - 1];
    const uint32_t kmax_r = r == 0 ? kmax[0] : kmax[NR - 1];
    const uint32_t klo_r = filt ? (r == 0 ? klo[0] : klo[NR - 1]) : 0u;
    const double zfull_r = r == 0 ? zfull[0] : zfull[NR - 1];
    const bool rbad_r = r == 0 ? rbad[0] : rbad[NR - 1];
    RowStat rs;
    rs.m = m_r;
    rs.kmax = kmax_r;
    rs.kstar = 0u;
    rs.cstar = 0u;
    rs.tie_total = 0u;
    rs.tie_cut = V;
    rs.zkept = zfull_r;
    rs.all_kept = 1;
    rs.bad = rbad_r ? 1 : 0;
    rs.partial = 0;
    uint32_t need_fb = 0u;
    if (!any_bad && filt) {
      rs.all_kept = 0;
      const int nbins = static_cast<int>(kmax_r - klo_r) + 1;
      if (!cut_scan_warp<DT, CS>(sh, r, hist + 4u * r * kWindow, nbins, rs, a.top_k, a.top_p, zfull_r, cexp))
        need_fb = 1u;
    }
    rs.inv_z = 1.f / static_cast<float>(rs.zkept);
    rs.thr = H::thr_pack(E::bits_of_key(rs.kstar));
    if (lane == 0) { sh.rs[r] = rs; sh.fb_need[r] = need_fb; }
  }
  __syncthreads();

  // ---------------- exact fallback: bitwise search of the cut over the keys
  {
    uint32_t slot = 0;
#pragma unroll 1
    for (int r = 0; r < NR; ++r) {
      if (!sh.fb_need[r]) continue;  // identical in every CTA of the cluster
      fallback_row<DT, CS>(cluster, sh, r == 0 ? buf[0] : buf[NR - 1], n, nvec, r, a.top_k, a.top_p,
                           r == 0 ? zfull[0] : zfull[NR - 1], cexp, slot);
    }
  }

  // ------ phase 3c: where a partial tie stops (only rows with a partial tie)
  bool part_any = false, part_fb = false;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    part_any |= sh.rs[r].partial != 0;
    part_fb |= sh.rs[r].partial != 0 && sh.fb_need[r] != 0;
  }
  if (part_any) tie_cuts<DT, CS, NR>(cluster, sh, buf[0], buf[NR - 1], hist, lo, hi, n, V, part_fb);
  const RowStat rp = sh.rs[0];
  const RowStat rq = sh.rs[NR - 1];

  // ----------------------------------------------- MODE_PROBS: write rows
  if (a.mode == MODE_PROBS) {
    write_probs<DT>(a, buf[0], rp, cexp, unit, lo, n, V);
    if (rp.bad && crank == 0 && tid == 0) set_status(a.status, SPEC_STATUS_BAD_ROW);
    cluster.sync();  // ------------------------------------------- sync: exit
    return;
  }

  const int kq = a.k;
  // ------------------------------------- phase 4: accept test at x_pos
  if constexpr (NR == 2) {
    const int x = a.tokens[static_cast<size_t>(b) * kq + pos];
    const bool x_ok = x >= 0 && x < V;
    UnitRec* rec = a.recs + unit;
    if (!x_ok || any_bad) {
      if (crank == 0 && tid == 0) {
        rec->accept = 0;
        rec->px = 0.f;
        rec->qx = 0.f;
        if (a.out_p) a.out_p[static_cast<size_t>(b) * kq + pos] = 0.f;
        if (a.out_q) a.out_q[static_cast<size_t>(b) * kq + pos] = 0.f;
        set_status(a.status, (!x_ok ? SPEC_STATUS_BAD_TOKEN : 0u) | (any_bad ? SPEC_STATUS_BAD_ROW : 0u));
        __threadfence();
        if (atomicAdd(a.tickets + b, 1u) == static_cast<uint32_t>(2 * kq)) sample_finalize(a, b);
      }
    } else if (x >= lo && x < hi && tid == 0) {
      const uint32_t bp = lds_elem<DT>(buf[0], x - lo), bq = lds_elem<DT>(buf[1], x - lo);
      const bool kp = kept_key(rp, E::key(bp), x);
      const bool kq2 = kept_key(rq, E::key(bq), x);
      const float px = kp ? softmax_mass(E::value(bp), rp.m, cexp) / static_cast<float>(rp.zkept) : 0.f;
      const float qx = kq2 ? softmax_mass(E::value(bq), rq.m, cexp) / static_cast<float>(rq.zkept) : 0.f;
      const float u = a.uniforms[static_cast<size_t>(b) * (kq + 2) + pos];
      rec->accept = (u * qx < px) ? 1 : 0;
      rec->px = px;
      rec->qx = qx;
      if (a.out_p) a.out_p[static_cast<size_t>(b) * kq + pos] = px;
      if (a.out_q) a.out_q[static_cast<size_t>(b) * kq + pos] = qx;
      __threadfence();
      if (atomicAdd(a.tickets + b, 1u) == static_cast<uint32_t>(2 * kq)) sample_finalize(a, b);
    }
  }

  // ------------------------- phase 5: residual (or bonus) inverse-CDF draw
  if (any_bad) {
    cluster.sync();  // ------------------------------------------- sync: exit
    if (crank == 0 && tid == 0) {
      a.recs[unit].drawn = -1;
      set_status(a.status, SPEC_STATUS_BAD_ROW);
      __threadfence();
      if (atomicAdd(a.tickets + b, 1u) == static_cast<uint32_t>(2 * kq)) sample_finalize(a, b);
    }
    return;
  }
  const float u_draw = a.uniforms[static_cast<size_t>(b) * (kq + 2) + (NR == 2 ? kq + 1 : kq)];
  bool use_q = NR == 2;
  double S = 0.0, Pc = 0.0;
  int owner = -1;
  for (int attempt = 0; attempt < 2; ++attempt) {
    float s = 0.f;
    for (int v = seg_beg + lane; v < seg_end; v += 32) {
      float w[8];
      const uint4 xp = lds128(buf[0] + 16u * v);
      const uint4 xq = use_q ? lds128(buf[NR - 1] + 16u * v) : xp;
      s += vec_weights<DT>(xp, xq, v * E::kPerVec, lo, n, use_q, rp, rq, cexp, w);
    }
    s = warp_sum_f32(s);
    if (lane == 0) sh.w_res[warp] = s;
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      for (int w = 0; w < kWarps; ++w) t += (double)sh.w_res[w];
      sh.x_res[attempt] = t;
    }
    cluster.sync();  // ---------------------------------------- sync: residual
    if (tid == 0) {  // total, owner CTA and its base, in fixed rank order
      double sc[CS], tot = 0.0, run = 0.0, pc = 0.0;
      int own = -1;
#pragma unroll
      for (int c = 0; c < CS; ++c) sc[c] = cluster.map_shared_rank(&sh, c)->x_res[attempt];
#pragma unroll
      for (int c = 0; c < CS; ++c) tot += sc[c];
      const double target = (double)u_draw * tot;
#pragma unroll
      for (int c = 0; c < CS; ++c) {
        if (own < 0 && sc[c] > 0.0 && run + sc[c] > target) { own = c; pc = run; }
        run += sc[c];
      }
      sh.b_S = tot;
      sh.b_Pc = pc;
      sh.b_owner = own;
    }
    __syncthreads();
    S = sh.b_S;
    if (S > 0.0 || !use_q) {
      owner = sh.b_owner;
      Pc = sh.b_Pc;
      break;
    }
    use_q = false;  // degenerate residual: draw from p instead
  }
  cluster.sync();  // ------------------------------------- sync: exit (no DSMEM after this)

  if (owner == crank)
    draw_walk<DT, NR>(a, sh, buf[0], buf[NR - 1], use_q, rp, rq, cexp, (double)u_draw * S - Pc, lo, n, unit, b);

}

template <int DT, int CS>
__global__ void __launch_bounds__(kThreads, 3) sample_kernel(const SampleArgs a) {
  using E = Elt<DT>;
  cg::cluster_group cluster = cg::this_cluster();
  const int unit = static_cast<int>(blockIdx.x) / CS;
  const int V = a.V;
  __shared__ Shm sh;
  extern __shared__ __align__(128) unsigned char dsm[];
  if (a.mode == MODE_SAMPLE) {
    const int b = unit / (a.k + 1);
    const int pos = unit % (a.k + 1);
    const unsigned char* rowp =
        static_cast<const unsigned char*>(a.target) + static_cast<size_t>(unit) * V * E::kBytes;
    if (pos < a.k) {
      const unsigned char* rowq = static_cast<const unsigned char*>(a.draft) +
                                  (static_cast<size_t>(b) * a.k + pos) * static_cast<size_t>(V) * E::kBytes;
      unit_body<DT, CS, 2>(a, cluster, sh, dsm, unit, b, pos, rowp, rowq);
    } else {
      unit_body<DT, CS, 1>(a, cluster, sh, dsm, unit, b, pos, rowp, nullptr);
    }
  } else {
    const unsigned char* rowp =
        static_cast<const unsigned char*>(a.target) + static_cast<size_t>(unit) * V * E::kBytes;
    unit_body<DT, CS, 1>(a, cluster, sh, dsm, unit, unit, 0, rowp, nullptr);
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

template <int DT, int CS>
static int launch_one(const SampleArgs& a, int units, size_t smem, cudaStream_t st) {
  auto kern = sample_kernel<DT, CS>;
  static size_t configured = 0;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    if (CS > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    configured = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units * CS));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

size_t sample_smem_bytes(int dtype, int chunk, bool filter) {
  const size_t es = dtype == DT_BF16 ? 2 : 4;
  const size_t buf = (chunk * es + 15) / 16 * 16;
  return 2 * buf + (filter ? 2 * kWindow * sizeof(uint32_t) : 0);
}

int launch_sample(const SampleArgs& a, int dtype, int cluster, int units, void* stream) {
  const bool filter = a.top_k > 0 || a.top_p < 1.f;
  const size_t smem = sample_smem_bytes(dtype, a.chunk, filter);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
#define SPECV_CASE(D, C) \
  if (dtype == D && cluster == C) return launch_one<D, C>(a, units, smem, st);
  SPECV_CASE(DT_BF16, 1) SPECV_CASE(DT_BF16, 2) SPECV_CASE(DT_BF16, 4) SPECV_CASE(DT_BF16, 8) SPECV_CASE(DT_BF16, 16)
  SPECV_CASE(DT_F32, 1) SPECV_CASE(DT_F32, 2) SPECV_CASE(DT_F32, 4) SPECV_CASE(DT_F32, 8) SPECV_CASE(DT_F32, 16)
#undef SPECV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace specv
