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
};

// ------------------------------------------------------------ row state

struct RowStat {
  float m;               // row maximum
  uint32_t kmax;         // key of m
  uint32_t kstar;        // kept iff key > kstar, or key == kstar and tie rank < cstar
  uint32_t cstar;
  uint32_t tie_total;    // tokens with key == kstar in the row
  uint32_t ties_before;  // such tokens in lower cluster ranks (partial rows only)
  uint32_t thr;          // packed threshold value of kstar (for the quick skip)
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
  double w_sum[kWarps][2];
  double w_res[kWarps];
  uint32_t w_tie[kWarps][2];
  double w_pm[kWarps];
  uint32_t w_pc[kWarps];
  uint32_t w_pk[kWarps];
  uint32_t fb_need[2];
  uint32_t owner_tie[2];
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

// Kept test for one element of a row.  `rank` is the element's rank among the
// tokens with key == kstar (consulted for partial rows only).
__device__ __forceinline__ bool kept_key(const RowStat& rs, uint32_t key, uint32_t rank) {
  if (rs.all_kept) return true;
  if (key > rs.kstar) return true;
  return key == rs.kstar && (!rs.partial || rank < rs.cstar);
}

// Draw weights of the elements of one 16-byte vector: w = max(0, p - q)
// (residual) or w = p (bonus).  tie_p / tie_q: rank of the vector's first
// kstar-valued element (partial rows only).  Vectors without an element at or
// above the target's cut value are skipped with one packed compare.
template <int DT>
__device__ __forceinline__ float vec_weights(const uint4& xp, const uint4& xq, int t0, int n, bool use_q,
                                             const RowStat& rp, const RowStat& rq, float cexp, uint32_t tie_p,
                                             uint32_t tie_q, float* w) {
  using E = Elt<DT>;
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < E::kPerVec; ++j) w[j] = 0.f;
  if (!rp.all_kept && !Hot<DT>::any_ge(xp, rp.thr)) return 0.f;
#pragma unroll
  for (int j = 0; j < E::kPerVec; ++j) {
    if (t0 + j < n) {
      const uint32_t bp = E::bits_of(xp, j);
      const uint32_t kp = E::key(bp);
      float pv = 0.f;
      if (kept_key(rp, kp, tie_p)) pv = softmax_mass(E::value(bp), rp.m, cexp) * rp.inv_z;
      if (rp.partial && kp == rp.kstar) ++tie_p;
      if (use_q) {
        const uint32_t bq = E::bits_of(xq, j);
        const uint32_t kq = E::key(bq);
        float qv = 0.f;
        if (kept_key(rq, kq, tie_q)) qv = softmax_mass(E::value(bq), rq.m, cexp) * rq.inv_z;
        if (rq.partial && kq == rq.kstar) ++tie_q;
        w[j] = fmaxf(pv - qv, 0.f);
      } else {
        w[j] = pv;
      }
      s += w[j];
    }
  }
  return s;
}

// Number of kstar-valued elements of a row in one vector.
template <int DT>
__device__ __forceinline__ uint32_t vec_ties(const uint4& x, int t0, int n, uint32_t kstar) {
  using E = Elt<DT>;
  uint32_t c = 0;
#pragma unroll
  for (int j = 0; j < E::kPerVec; ++j)
    if (t0 + j < n && E::key(E::bits_of(x, j)) == kstar) ++c;
  return c;
}

enum PassKind { PASS_COUNT_GE = 0, PASS_MASS_GT = 1, PASS_MIN_GE = 2, PASS_COUNT_EQ = 3 };

// One full pass over this CTA's slice of one row, reduced over the cluster.
// Used only by the exact fallback search of the cut.
template <int DT, int CS>
__device__ double cluster_pass(cg::cluster_group& cluster, Shm& sh, const uint4* buf, int n, int nvec, int kind,
                               uint32_t kappa, float m, float c, uint32_t& slot) {
  using E = Elt<DT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t cnt = 0, kmin = 0xFFFFFFFFu;
  float mass = 0.f;
  for (int v = tid; v < nvec; v += kThreads) {
    const uint4 x = buf[v];
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
  const double dm = warp_sum_f64((double)mass);
  cnt = warp_sum_u32(cnt);
  kmin = warp_min_u32(kmin);
  if (lane == 0) { sh.w_pm[warp] = dm; sh.w_pc[warp] = cnt; sh.w_pk[warp] = kmin; }
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

}  // namespace

__device__ void sample_finalize(const SampleArgs& a, int b);

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
  const uint4* buf[2] = {reinterpret_cast<const uint4*>(dsm), reinterpret_cast<const uint4*>(dsm + bufbytes)};
  uint32_t* hist = reinterpret_cast<uint32_t*>(dsm + 2 * bufbytes);
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
        bulk_copy_g2s(const_cast<uint4*>(buf[r]), rows[r] + static_cast<size_t>(lo) * E::kBytes,
                      static_cast<uint32_t>(n * E::kBytes), &sh.mbar);
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    if (!aligned[r]) {
      for (int t = tid; t < n; t += kThreads) {
        const uint32_t bits = E::bits_at(rows[r], static_cast<int64_t>(lo) + t);
        if (E::kBytes == 2) reinterpret_cast<uint16_t*>(const_cast<uint4*>(buf[r]))[t] = static_cast<uint16_t>(bits);
        else reinterpret_cast<uint32_t*>(const_cast<uint4*>(buf[r]))[t] = bits;
      }
    }
  }
  if (filt)
    for (int t = tid; t < NR * kWindow; t += kThreads) hist[t] = 0u;
  if (!mbar_wait_bounded(&sh.mbar, 0)) set_status(a.status, SPEC_STATUS_TIMEOUT);
  __syncthreads();

  // ------------------------------------------------------ phase 1: max
  {
    typename H::MaxAcc st[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) H::max_init(st[r]);
    for (int v = tid; v < nfull; v += kThreads) {
#pragma unroll
      for (int r = 0; r < NR; ++r) H::max_vec(buf[r][v], st[r]);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      float mx = H::max_finish(st[r]);
      for (int t = nfull * E::kPerVec + tid; t < n; t += kThreads) mx = max_nan(mx, E::value(E::bits_at(buf[r], t)));
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
          H::mass_vec(buf[r][v], m2, c2, acc0);
          H::mass_vec(buf[r][v + kThreads], m2, c2, acc1);
        }
        if (v < nfull) H::mass_vec(buf[r][v], m2, c2, acc0);
        float s0, s1, s2, s3;
        upk(acc0, s0, s1);
        upk(acc1, s2, s3);
        float s = (s0 + s1) + (s2 + s3);
        for (int t = nfull * E::kPerVec + tid; t < n; t += kThreads)
          s += softmax_mass(E::value(E::bits_at(buf[r], t)), m[r], cexp);
        const double ws = warp_sum_f64((double)s);
        if (lane == 0) sh.w_sum[warp][r] = ws;
      }
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        double s = 0.0;
        if (!any_bad)
          for (int w = 0; w < kWarps; ++w) s += sh.w_sum[w][r];
        sh.x_sum[r] = s;
      }
    }
    cluster.sync();  // -------------------------------------------- sync: sum
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      double v = 0.0;
      if (lane < CS) v = cluster.map_shared_rank(&sh, lane)->x_sum[r];
      zfull[r] = cluster_sum_f64<CS>(v);
    }
  }

  // ------------------------- phase 3: exact-value histogram near the top
  // Bins d = kmax - key count the tokens of one value each.  Only tokens that
  // can survive the cut are counted: at most kWindow values below the max,
  // and with top-p alone no token whose mass is below (1 - top_p) Z / V (all
  // tokens ranked at or below such a token weigh less than (1 - top_p) Z, so
  // the mass ranked before it exceeds top_p Z).  Half of that bound is used,
  // as margin for rounding.
  uint32_t klo[NR];
  if (filt) {
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      uint32_t kl = kmax[r] >= static_cast<uint32_t>(kWindow - 1) ? kmax[r] - static_cast<uint32_t>(kWindow - 1) : 0u;
      const uint32_t kninf = E::key(E::kBytes == 2 ? 0xFF80u : 0xFF800000u);  // -inf
      if (kl < kninf) kl = kninf;
      if (topp_on && !topk_on && !any_bad && zfull[r] > 0.0) {
        const double lim = 0.5 * (1.0 - (double)a.top_p) * zfull[r] / (double)V;
        const float vb = m[r] + static_cast<float>(log2(lim)) / cexp;
        if (isfinite(vb) && vb > -3.0e38f) {
          const uint32_t kb = E::key(bits_round_down<DT>(vb));
          if (kb > kl) kl = kb;
        }
      }
      klo[r] = kl;
    }
    if (!any_bad) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const uint32_t thr = H::thr_pack(E::bits_of_key(klo[r]));
        uint32_t* hr = hist + r * kWindow;
        const uint32_t km = kmax[r];
        for (int v = tid; v < nfull; v += kThreads) {
          const uint4 x = buf[r][v];
          if (!H::any_ge(x, thr)) continue;
          uint32_t msk = H::mask_ge(x, thr);
          while (msk) {
            const int j = __ffs(msk) - 1;
            msk &= msk - 1u;
            atomicAdd(hr + (km - E::key(E::bits_of(x, j))), 1u);
          }
        }
        for (int t = nfull * E::kPerVec + tid; t < n; t += kThreads) {
          const uint32_t k = E::key(E::bits_at(buf[r], t));
          if (k >= klo[r]) atomicAdd(hr + (km - k), 1u);
        }
      }
    }
    __syncthreads();
    cluster.sync();  // ---------------------------------------- sync: histogram
  }

  // ------------------------------------ phase 3b: the kept set of each row
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
    rs.ties_before = 0u;
    rs.thr = 0u;
    rs.zkept = zfull_r;
    rs.all_kept = 1;
    rs.bad = rbad_r ? 1 : 0;
    rs.partial = 0;
    uint32_t need_fb = 0u;
    if (!any_bad && filt) {
      rs.all_kept = 0;
      const float mr = m_r;
      const int nbins = static_cast<int>(kmax_r - klo_r) + 1;
      auto bin = [&](int d) -> uint32_t {
        if (d >= nbins) return 0u;
        uint32_t c = 0;
#pragma unroll
        for (int q = 0; q < CS; ++q) c += cluster.map_shared_rank(hist, q)[r * kWindow + d];
        return c;
      };
      auto bin_mass = [&](int d) -> float {
        return softmax_mass(value_of_key<DT>(kmax_r - static_cast<uint32_t>(d)), mr, cexp);
      };
      bool ok = true;
      uint32_t dk = 0, ck = 0, tk = 0;
      double zk = zfull_r;
      if (topk_on) {
        ok = false;
        uint32_t base = 0;
        double mbase = 0.0;
        for (int d0 = 0; d0 < nbins; d0 += 32) {
          const int d = d0 + lane;
          const uint32_t cnt = bin(d);
          const float ed = cnt ? bin_mass(d) : 0.f;
          const double ms = cnt ? (double)cnt * (double)ed : 0.0;
          const uint32_t incl = warp_incl_scan_u32(cnt);
          const double mincl = warp_incl_scan_f64(ms);
          const unsigned ball = __ballot_sync(kFull, base + incl >= static_cast<uint32_t>(a.top_k));
          if (ball) {
            const int l = __ffs(ball) - 1;
            dk = static_cast<uint32_t>(d0 + l);
            const uint32_t before = base + __shfl_sync(kFull, incl - cnt, l);
            ck = static_cast<uint32_t>(a.top_k) - before;
            tk = __shfl_sync(kFull, cnt, l);
            const double mb = mbase + __shfl_sync(kFull, mincl - ms, l);
            zk = mb + (double)ck * (double)__shfl_sync(kFull, ed, l);
            ok = true;
            break;
          }
          base += __shfl_sync(kFull, incl, 31);
          mbase += __shfl_sync(kFull, mincl, 31);
        }
      }
      uint32_t dstar = dk, cstar = ck, tstar = tk;
      double zkept = zk;
      if (ok && topp_on) {
        ok = false;
        const double target = (double)a.top_p * zk;
        double mbase = 0.0;
        for (int d0 = 0; d0 < nbins; d0 += 32) {
          const int d = d0 + lane;
          const uint32_t real = bin(d);
          uint32_t cnt = real;
          if (topk_on && static_cast<uint32_t>(d) > dk) cnt = 0;
          if (topk_on && static_cast<uint32_t>(d) == dk) cnt = ck;
          const float ed = cnt ? bin_mass(d) : 0.f;
          const double ms = cnt ? (double)cnt * (double)ed : 0.0;
          const double mincl = warp_incl_scan_f64(ms);
          const unsigned ball = __ballot_sync(kFull, cnt > 0 && mbase + mincl >= target);
          if (ball) {
            const int l = __ffs(ball) - 1;
            dstar = static_cast<uint32_t>(d0 + l);
            const double mb = mbase + __shfl_sync(kFull, mincl - ms, l);
            const uint32_t avail = __shfl_sync(kFull, cnt, l);
            const float ep = __shfl_sync(kFull, ed, l);
            tstar = __shfl_sync(kFull, real, l);
            const double xneed = (target - mb) / (double)ep;
            uint32_t cp = avail;
            if (xneed < (double)avail) cp = max(1u, static_cast<uint32_t>(ceil(xneed)));
            cstar = cp;
            zkept = mb + (double)cp * (double)ep;
            ok = true;
            break;
          }
          mbase += __shfl_sync(kFull, mincl, 31);
          if (topk_on && static_cast<uint32_t>(d0 + 31) >= dk) break;
        }
      }
      if (ok) {
        rs.kstar = rs.kmax - dstar;
        rs.cstar = cstar;
        rs.tie_total = tstar;
        rs.zkept = zkept;
        rs.partial = cstar < tstar ? 1 : 0;
      } else {
        need_fb = 1u;
      }
    }
    rs.inv_z = static_cast<float>(1.0 / rs.zkept);
    rs.thr = H::thr_pack(E::bits_of_key(rs.kstar));
    if (lane == 0) { sh.rs[r] = rs; sh.fb_need[r] = need_fb; }
  }
  __syncthreads();

  // ---------------- exact fallback: bitwise search of the cut over the keys
  {
    uint32_t slot = 0;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      if (!sh.fb_need[r]) continue;  // identical in every CTA of the cluster
      RowStat rs = sh.rs[r];
      const uint4* bb = buf[r];
      const int kb = E::kKeyBits;
      uint32_t kk = 0, ck = 0, tk = 0;
      double zk = zfull[r];
      if (topk_on) {
        for (int bit = kb - 1; bit >= 0; --bit) {
          const uint32_t cand = kk | (1u << bit);
          const double cnt = cluster_pass<DT, CS>(cluster, sh, bb, n, nvec, PASS_COUNT_GE, cand, rs.m, cexp, slot);
          if (cnt >= (double)a.top_k) kk = cand;
        }
        const uint32_t gt = (kk == 0xFFFFFFFFu) ? 0u
            : static_cast<uint32_t>(cluster_pass<DT, CS>(cluster, sh, bb, n, nvec, PASS_COUNT_GE, kk + 1u, rs.m, cexp, slot));
        ck = static_cast<uint32_t>(a.top_k) - gt;
        tk = static_cast<uint32_t>(cluster_pass<DT, CS>(cluster, sh, bb, n, nvec, PASS_COUNT_EQ, kk, rs.m, cexp, slot));
        const float ek = softmax_mass(value_of_key<DT>(kk), rs.m, cexp);
        zk = cluster_pass<DT, CS>(cluster, sh, bb, n, nvec, PASS_MASS_GT, kk, rs.m, cexp, slot) + (double)ck * (double)ek;
      }
      uint32_t kstar = kk, cstar = ck, tstar = tk;
      double zkept = zk;
      if (topp_on) {
        const double target = (double)a.top_p * zk;
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
      rs.inv_z = static_cast<float>(1.0 / zkept);
      rs.thr = H::thr_pack(E::bits_of_key(kstar));
      __syncthreads();
      if (tid == 0) sh.rs[r] = rs;
      __syncthreads();
    }
  }

  // ------------------- phase 3c: tie ranks, only for rows with a partial tie
  bool part_any = false;
#pragma unroll
  for (int r = 0; r < NR; ++r) part_any |= sh.rs[r].partial != 0;
  uint32_t warp_tie_base[2] = {0u, 0u};
  if (part_any) {
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      uint32_t c = 0;
      if (sh.rs[r].partial)
        for (int v = seg_beg + lane; v < seg_end; v += 32) c += vec_ties<DT>(buf[r][v], v * E::kPerVec, n, sh.rs[r].kstar);
      c = warp_sum_u32(c);
      if (lane == 0) sh.w_tie[warp][r] = c;
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        uint32_t s = 0;
        for (int w = 0; w < kWarps; ++w) s += sh.w_tie[w][r];
        sh.x_tie[r] = s;
      }
    }
    cluster.sync();  // --------------------------------------------- sync: ties
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      uint32_t before = 0;
      for (int q = 0; q < crank; ++q) before += cluster.map_shared_rank(&sh, q)->x_tie[r];
      uint32_t wb = 0;
      for (int w = 0; w < warp; ++w) wb += sh.w_tie[w][r];
      warp_tie_base[r] = before + wb;
      if (tid == 0) sh.rs[r].ties_before = before;
    }
    __syncthreads();
  }
  const RowStat rp = sh.rs[0];
  const RowStat rq = sh.rs[NR - 1];

  // ----------------------------------------------- MODE_PROBS: write rows
  if (a.mode == MODE_PROBS) {
    float* out = a.out_probs + static_cast<size_t>(unit) * V + lo;
    const bool vec_out = ((reinterpret_cast<uintptr_t>(out) & 15u) == 0) && (V % 4 == 0);
    uint32_t run = warp_tie_base[0];
    for (int it = 0; it < seg_iters; ++it) {
      const int v = seg_beg + it * 32 + lane;
      const bool valid = v < seg_end;
      const int t0 = v * E::kPerVec;
      const uint4 x = valid ? buf[0][v] : make_uint4(0u, 0u, 0u, 0u);
      uint32_t base = 0;
      if (rp.partial) {
        const uint32_t c = valid ? vec_ties<DT>(x, t0, n, rp.kstar) : 0u;
        const uint32_t incl = warp_incl_scan_u32(c);
        base = run + incl - c;
        run += __shfl_sync(kFull, incl, 31);
      }
      if (valid) {
        float w[8];
        vec_weights<DT>(x, x, t0, n, false, rp, rp, cexp, base, base, w);
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
    } else if (x >= lo && x < hi) {
      if (part_any) {  // tie ranks of x inside this CTA
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          uint32_t c = 0;
          if (sh.rs[r].partial)
            for (int t = tid; t < x - lo; t += kThreads) c += (E::key(E::bits_at(buf[r], t)) == sh.rs[r].kstar);
          c = warp_sum_u32(c);
          if (lane == 0) sh.w_tie[warp][r] = c;
        }
        __syncthreads();
        if (tid == 0)
          for (int r = 0; r < 2; ++r) {
            uint32_t s = sh.rs[r].ties_before;
            for (int w = 0; w < kWarps; ++w) s += sh.w_tie[w][r];
            sh.owner_tie[r] = s;
          }
        __syncthreads();
      }
      if (tid == 0) {
        const uint32_t bp = E::bits_at(buf[0], x - lo), bq = E::bits_at(buf[1], x - lo);
        const bool kp = kept_key(rp, E::key(bp), part_any ? sh.owner_tie[0] : 0u);
        const bool kq2 = kept_key(rq, E::key(bq), part_any ? sh.owner_tie[1] : 0u);
        const double px = kp ? (double)softmax_mass(E::value(bp), rp.m, cexp) / rp.zkept : 0.0;
        const double qx = kq2 ? (double)softmax_mass(E::value(bq), rq.m, cexp) / rq.zkept : 0.0;
        const double u = (double)a.uniforms[static_cast<size_t>(b) * (kq + 2) + pos];
        rec->accept = (u * qx < px) ? 1 : 0;
        rec->px = static_cast<float>(px);
        rec->qx = static_cast<float>(qx);
        if (a.out_p) a.out_p[static_cast<size_t>(b) * kq + pos] = static_cast<float>(px);
        if (a.out_q) a.out_q[static_cast<size_t>(b) * kq + pos] = static_cast<float>(qx);
        __threadfence();
        if (atomicAdd(a.tickets + b, 1u) == static_cast<uint32_t>(2 * kq)) sample_finalize(a, b);
      }
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
    if (!part_any) {
      for (int v = seg_beg + lane; v < seg_end; v += 32) {
        float w[8];
        s += vec_weights<DT>(buf[0][v], use_q ? buf[NR - 1][v] : buf[0][v], v * E::kPerVec, n, use_q, rp, rq, cexp,
                             0u, 0u, w);
      }
    } else {
      uint32_t runp = warp_tie_base[0], runq = warp_tie_base[1];
      for (int it = 0; it < seg_iters; ++it) {
        const int v = seg_beg + it * 32 + lane;
        const bool valid = v < seg_end;
        const int t0 = v * E::kPerVec;
        const uint4 xp = valid ? buf[0][v] : make_uint4(0u, 0u, 0u, 0u);
        const uint4 xq = (valid && use_q) ? buf[NR - 1][v] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t cp = (valid && rp.partial) ? vec_ties<DT>(xp, t0, n, rp.kstar) : 0u;
        const uint32_t cq = (valid && use_q && rq.partial) ? vec_ties<DT>(xq, t0, n, rq.kstar) : 0u;
        const uint32_t ip = warp_incl_scan_u32(cp), iq = warp_incl_scan_u32(cq);
        const uint32_t bp = runp + ip - cp, bq = runq + iq - cq;
        runp += __shfl_sync(kFull, ip, 31);
        runq += __shfl_sync(kFull, iq, 31);
        if (valid) {
          float w[8];
          s += vec_weights<DT>(xp, xq, t0, n, use_q, rp, rq, cexp, bp, bq, w);
        }
      }
    }
    const double ws = warp_sum_f64((double)s);
    if (lane == 0) sh.w_res[warp] = ws;
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      for (int w = 0; w < kWarps; ++w) t += sh.w_res[w];
      sh.x_res[attempt] = t;
    }
    cluster.sync();  // ---------------------------------------- sync: residual
    double mine = 0.0;
    if (lane < CS) mine = cluster.map_shared_rank(&sh, lane)->x_res[attempt];
    S = cluster_sum_f64<CS>(mine);
    if (S > 0.0 || !use_q) {
      const double target = (double)u_draw * S;
      double run = 0.0;
      for (int c = 0; c < CS; ++c) {
        const double sc = __shfl_sync(kFull, mine, c);
        if (owner < 0 && sc > 0.0 && run + sc > target) { owner = c; Pc = run; }
        run += sc;
      }
      break;
    }
    use_q = false;  // degenerate residual: draw from p instead
  }
  cluster.sync();  // ------------------------------------- sync: exit (no DSMEM after this)

  if (owner == crank) {
    const double target = (double)u_draw * S - Pc;
    if (tid == 0) {
      double run = 0.0, wbase = 0.0, lbase = 0.0;
      int wsel = -1, wlast = -1;
      for (int w = 0; w < kWarps; ++w) {
        const double sw = sh.w_res[w];
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
      uint32_t runp = warp_tie_base[0], runq = warp_tie_base[1];
      for (int it = 0; it < seg_iters && token < 0; ++it) {
        const int v = seg_beg + it * 32 + lane;
        const bool valid = v < seg_end;
        const int t0 = v * E::kPerVec;
        const uint4 xp = valid ? buf[0][v] : make_uint4(0u, 0u, 0u, 0u);
        const uint4 xq = (valid && use_q) ? buf[NR - 1][v] : make_uint4(0u, 0u, 0u, 0u);
        uint32_t bp = 0, bq = 0;
        if (part_any) {
          const uint32_t cp = (valid && rp.partial) ? vec_ties<DT>(xp, t0, n, rp.kstar) : 0u;
          const uint32_t cq = (valid && use_q && rq.partial) ? vec_ties<DT>(xq, t0, n, rq.kstar) : 0u;
          const uint32_t ip = warp_incl_scan_u32(cp), iq = warp_incl_scan_u32(cq);
          bp = runp + ip - cp;
          bq = runq + iq - cq;
          runp += __shfl_sync(kFull, ip, 31);
          runq += __shfl_sync(kFull, iq, 31);
        }
        float w[8];
        float ls = 0.f;
        int lpos = -1;
        if (valid) {
          ls = vec_weights<DT>(xp, xq, t0, n, use_q, rp, rq, cexp, bp, bq, w);
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
}

template <int DT, int CS>
__global__ void __launch_bounds__(kThreads) sample_kernel(const SampleArgs a) {
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
