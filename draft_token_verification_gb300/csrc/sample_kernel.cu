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
// read from HBM exactly once.  The row statistics (max, sum of masses, an
// exact-value histogram of the top of the row for the top-k / top-p cut) are
// combined across the cluster through distributed shared memory.  The accept
// test is done by the CTA that holds x_i; the residual (or bonus) draw is
// done speculatively for every unit, so no row is read twice; the CTA that
// holds the drawn token writes it.  The last writer of a sequence (atomic
// ticket, no spin-wait) applies the first-rejection rule and commits.
#include <cuda_runtime.h>
#include <math.h>

#include "device_common.cuh"

namespace specv {

namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;

struct RowStat {
  float m;               // row maximum
  uint32_t kmax;         // key of m
  uint32_t kstar;        // kept iff key > kstar, or key == kstar and tie rank < cstar
  uint32_t cstar;
  uint32_t tie_total;    // tokens with key == kstar in the row
  uint32_t ties_before;  // such tokens in lower cluster ranks (partial rows only)
  double zkept;          // sum of masses over the kept set
  float inv_z;
  int all_kept;
  int bad;
  int partial;           // 0 < cstar < tie_total
};

struct Shm {
  // exchange slots, read by the other CTAs of the cluster
  float x_max[2];
  uint32_t x_bad[2];
  double x_sum[2];
  uint32_t x_tie[2];
  double x_res[2];
  double x_pm[2];
  uint32_t x_pc[2];
  uint32_t x_pk[2];
  // CTA scratch
  float w_max[kWarps][2];
  uint32_t w_bad[kWarps][2];
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

// Fixed-order sum of one double per cluster rank (every lane gets the total).
template <int CS>
__device__ __forceinline__ double cluster_sum_f64(double mine_lane_c) {
  double z = 0.0;
#pragma unroll
  for (int c = 0; c < CS; ++c) z += __shfl_sync(kFull, mine_lane_c, c);
  return z;
}

// Kept test for one element of a row.  `rank` is the element's rank among the
// tokens with key == kstar (only consulted for partial rows).
__device__ __forceinline__ bool kept_key(const RowStat& rs, uint32_t key, uint32_t rank) {
  if (rs.all_kept) return true;
  if (key > rs.kstar) return true;
  return key == rs.kstar && (!rs.partial || rank < rs.cstar);
}

// Per-vector evaluation of the draw weight w_t (residual max(0, p - q) or p)
// for the elements of one 16-byte vector of each row.  tie_p / tie_q are the
// ranks of this vector's first kstar-valued element (partial rows only).
template <int DT>
__device__ __forceinline__ void draw_weights(const uint4& xp, const uint4& xq, int t0, int n, bool use_q,
                                             const RowStat& rp, const RowStat& rq, float cp, float cq,
                                             uint32_t tie_p, uint32_t tie_q, float* w) {
  using E = Elt<DT>;
#pragma unroll
  for (int j = 0; j < E::kPerVec; ++j) {
    w[j] = 0.f;
    if (t0 + j < n) {
      const uint32_t bp = E::bits_of(xp, j);
      const uint32_t kp = E::key(bp);
      float pv = 0.f;
      if (kept_key(rp, kp, tie_p)) pv = softmax_mass(E::value(bp), rp.m, cp) * rp.inv_z;
      if (rp.partial && kp == rp.kstar) ++tie_p;
      if (use_q) {
        const uint32_t bq = E::bits_of(xq, j);
        const uint32_t kq = E::key(bq);
        float qv = 0.f;
        if (kept_key(rq, kq, tie_q)) qv = softmax_mass(E::value(bq), rq.m, cq) * rq.inv_z;
        if (rq.partial && kq == rq.kstar) ++tie_q;
        w[j] = fmaxf(pv - qv, 0.f);
      } else {
        w[j] = pv;
      }
    }
  }
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

// Reduction of one value over the CTA (thread 0 gets it).
enum PassKind { PASS_COUNT_GE = 0, PASS_MASS_GT = 1, PASS_MIN_GE = 2, PASS_COUNT_EQ = 3 };

// One full pass over this CTA's slice of one row, reduced over the cluster.
// Used only by the exact fallback search (rows whose cut lies outside the
// histogram window, and fp32 rows).
template <int DT, int CS>
__device__ double cluster_pass(cg::cluster_group& cluster, Shm& sh, const uint4* buf, int n, int nvec,
                               int kind, uint32_t kappa, float m, float c, uint32_t& slot) {
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
  double dm = warp_sum_f64((double)mass);
  cnt = warp_sum_u32(cnt);
  kmin = warp_min_u32(kmin);
  if (lane == 0) { sh.w_pm[warp] = dm; sh.w_pc[warp] = cnt; sh.w_pk[warp] = kmin; }
  __syncthreads();
  if (tid == 0) {
    double tm = 0.0; uint32_t tc = 0, tk = 0xFFFFFFFFu;
    for (int w = 0; w < kWarps; ++w) { tm += sh.w_pm[w]; tc += sh.w_pc[w]; tk = min(tk, sh.w_pk[w]); }
    sh.x_pm[s] = tm; sh.x_pc[s] = tc; sh.x_pk[s] = tk;
  }
  cluster.sync();
  double res;
  {
    double vm = 0.0; uint32_t vc = 0, vk = 0xFFFFFFFFu;
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

}  // namespace

__device__ void sample_finalize(const SampleArgs& a, int b);

template <int DT, int CS>
__global__ void __launch_bounds__(kThreads) sample_kernel(const SampleArgs a) {
  using E = Elt<DT>;
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = static_cast<int>(cluster.block_rank());
  const int unit = static_cast<int>(blockIdx.x) / CS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;
  __shared__ Shm sh;
  extern __shared__ __align__(128) unsigned char dsm[];

  // ------------------------------------------------------------ the unit
  int b, pos;
  bool has_q;
  const unsigned char* rowp;
  const unsigned char* rowq = nullptr;
  if (a.mode == MODE_SAMPLE) {
    b = unit / (a.k + 1);
    pos = unit % (a.k + 1);
    has_q = pos < a.k;
    rowp = static_cast<const unsigned char*>(a.target) + static_cast<size_t>(unit) * V * E::kBytes;
    if (has_q)
      rowq = static_cast<const unsigned char*>(a.draft) +
             (static_cast<size_t>(b) * a.k + pos) * static_cast<size_t>(V) * E::kBytes;
  } else {
    b = unit;
    pos = 0;
    has_q = false;
    rowp = static_cast<const unsigned char*>(a.target) + static_cast<size_t>(unit) * V * E::kBytes;
  }
  const int nrows = has_q ? 2 : 1;
  const float T = a.temperature_per_seq ? a.temperature_per_seq[b] : a.temperature;
  const bool bad_t = !(T > 0.f) || isinf(T);
  const float cexp = kLog2e / T;

  const int lo = min(V, crank * a.chunk);
  const int hi = min(V, lo + a.chunk);
  const int n = hi - lo;
  const int nvec = (n * E::kBytes + 15) / 16;
  const int bufbytes = ((a.chunk * E::kBytes + 15) / 16) * 16;
  uint4* buf[2] = {reinterpret_cast<uint4*>(dsm), reinterpret_cast<uint4*>(dsm + bufbytes)};
  uint32_t* hist = reinterpret_cast<uint32_t*>(dsm + 2 * bufbytes);

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
  const bool al[2] = {a.aligned_target != 0, a.aligned_draft != 0};
  const unsigned char* rows[2] = {rowp, rowq};
  if (tid == 0) {
    uint32_t tx = 0;
    for (int r = 0; r < nrows; ++r)
      if (al[r] && n > 0) tx += static_cast<uint32_t>(n * E::kBytes);
    mbar_arrive_expect_tx(&sh.mbar, tx);
    for (int r = 0; r < nrows; ++r)
      if (al[r] && n > 0)
        bulk_copy_g2s(buf[r], rows[r] + static_cast<size_t>(lo) * E::kBytes, static_cast<uint32_t>(n * E::kBytes),
                      &sh.mbar);
  }
  for (int r = 0; r < nrows; ++r) {
    if (!al[r]) {
      for (int t = tid; t < n; t += kThreads) {
        const uint32_t bits = E::bits_at(rows[r], static_cast<int64_t>(lo) + t);
        if (E::kBytes == 2) reinterpret_cast<uint16_t*>(buf[r])[t] = static_cast<uint16_t>(bits);
        else reinterpret_cast<uint32_t*>(buf[r])[t] = bits;
      }
    }
  }
  if (filt)
    for (int t = tid; t < 2 * kWindow; t += kThreads) hist[t] = 0u;
  if (!mbar_wait_bounded(&sh.mbar, 0)) set_status(a.status, SPEC_STATUS_TIMEOUT);
  __syncthreads();

  // ------------------------------------------------------ phase 1: max
  {
    float mx[2] = {-INFINITY, -INFINITY};
    uint32_t bad[2] = {0u, 0u};
    for (int v = tid; v < nvec; v += kThreads) {
      const int t0 = v * E::kPerVec;
      for (int r = 0; r < nrows; ++r) {
        const uint4 x = buf[r][v];
#pragma unroll
        for (int j = 0; j < E::kPerVec; ++j) {
          if (t0 + j < n) {
            const uint32_t bits = E::bits_of(x, j);
            const float val = E::value(bits);
            if (E::nonfinite_or_nan(bits) && !(val == -INFINITY)) bad[r] = 1u;
            mx[r] = fmaxf(mx[r], val);
          }
        }
      }
    }
    for (int r = 0; r < nrows; ++r) {
      const float wm = warp_max(mx[r]);
      const uint32_t wb = warp_max_u32(bad[r]);
      if (lane == 0) { sh.w_max[warp][r] = wm; sh.w_bad[warp][r] = wb; }
    }
    __syncthreads();
    if (tid == 0) {
      for (int r = 0; r < nrows; ++r) {
        float m = -INFINITY; uint32_t bd = 0;
        for (int w = 0; w < kWarps; ++w) { m = fmaxf(m, sh.w_max[w][r]); bd |= sh.w_bad[w][r]; }
        sh.x_max[r] = m; sh.x_bad[r] = bd;
      }
    }
  }
  cluster.sync();  // ---------------------------------------------- sync 1
  float m[2] = {-INFINITY, -INFINITY};
  bool rbad[2] = {true, true};
  uint32_t kmax[2] = {0u, 0u};
  for (int r = 0; r < nrows; ++r) {
    float pm = -INFINITY; uint32_t pb = 0;
    if (lane < CS) {
      const Shm* peer = cluster.map_shared_rank(&sh, lane);
      pm = peer->x_max[r]; pb = peer->x_bad[r];
    }
    m[r] = warp_max(pm);
    pb = warp_max_u32(pb);
    rbad[r] = pb != 0u || m[r] == -INFINITY || bad_t;
    const uint32_t mbits = (E::kBytes == 2) ? (__float_as_uint(m[r]) >> 16) : __float_as_uint(m[r]);
    kmax[r] = E::key(mbits);
  }
  const bool any_bad = rbad[0] || (has_q && rbad[1]);

  // ----------------------------------- phase 2: masses and the cut histogram
  const bool need_sum = !topk_on;
  if (!any_bad) {
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int v = tid; v < nvec; v += kThreads) {
      const int t0 = v * E::kPerVec;
      for (int r = 0; r < nrows; ++r) {
        const uint4 x = buf[r][v];
#pragma unroll
        for (int j = 0; j < E::kPerVec; ++j) {
          if (t0 + j < n) {
            const uint32_t bits = E::bits_of(x, j);
            if (need_sum) acc[r][j & 3] += softmax_mass(E::value(bits), m[r], cexp);
            if (filt) {
              const uint32_t d = kmax[r] - E::key(bits);
              if (d < static_cast<uint32_t>(kWindow)) atomicAdd(&hist[r * kWindow + d], 1u);
            }
          }
        }
      }
    }
    for (int r = 0; r < nrows; ++r) {
      const double s = warp_sum_f64((double)((acc[r][0] + acc[r][1]) + (acc[r][2] + acc[r][3])));
      if (lane == 0) sh.w_sum[warp][r] = s;
    }
  }
  __syncthreads();
  if (tid == 0) {
    for (int r = 0; r < nrows; ++r) {
      double s = 0.0;
      if (!any_bad)
        for (int w = 0; w < kWarps; ++w) s += sh.w_sum[w][r];
      sh.x_sum[r] = s;
    }
  }
  cluster.sync();  // ---------------------------------------------- sync 2
  double zfull[2] = {0.0, 0.0};
  for (int r = 0; r < nrows; ++r) {
    double v = 0.0;
    if (lane < CS) v = cluster.map_shared_rank(&sh, lane)->x_sum[r];
    zfull[r] = cluster_sum_f64<CS>(v);
  }

  // ------------------------------------ phase 2b: the kept set of each row
  if (warp < nrows) {
    const int r = warp;
    RowStat rs;
    rs.m = m[r];
    rs.kmax = kmax[r];
    rs.kstar = 0u;
    rs.cstar = 0u;
    rs.tie_total = 0u;
    rs.ties_before = 0u;
    rs.zkept = zfull[r];
    rs.all_kept = 1;
    rs.bad = rbad[r] ? 1 : 0;
    rs.partial = 0;
    uint32_t need_fb = 0u;
    if (!any_bad && filt) {
      rs.all_kept = 0;
      const float mr = m[r];
      // cluster-wide count of bin d (every lane a different bin)
      auto bin = [&](int d) -> uint32_t {
        uint32_t c = 0;
#pragma unroll
        for (int q = 0; q < CS; ++q) c += cluster.map_shared_rank(hist, q)[r * kWindow + d];
        return c;
      };
      auto bin_mass = [&](int d) -> float {
        const uint32_t kk = rs.kmax - static_cast<uint32_t>(d);
        return softmax_mass(value_of_key<DT>(kk), mr, cexp);
      };
      bool ok = true;
      uint32_t dk = 0, ck = 0, tk = 0;
      double zk = zfull[r];
      if (topk_on) {
        ok = false;
        uint32_t base = 0;
        double mbase = 0.0;
        for (int d0 = 0; d0 < kWindow; d0 += 32) {
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
        for (int d0 = 0; d0 < kWindow; d0 += 32) {
          const int d = d0 + lane;
          uint32_t real = bin(d);
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
    if (lane == 0) { sh.rs[r] = rs; sh.fb_need[r] = need_fb; }
  }
  __syncthreads();

  // ---------------- exact fallback: bitwise search of the cut over the keys
  uint32_t slot = 0;
  for (int r = 0; r < nrows; ++r) {
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
      // G(kappa): mass of the top-k set above kappa
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
    __syncthreads();
    if (tid == 0) sh.rs[r] = rs;
    __syncthreads();
  }

  // ------------------- phase 2c: tie ranks, only for rows with a partial tie
  const bool part_any = sh.rs[0].partial || (has_q && sh.rs[1].partial);
  uint32_t warp_tie_base[2] = {0u, 0u};
  if (part_any) {
    for (int r = 0; r < nrows; ++r) {
      uint32_t c = 0;
      if (sh.rs[r].partial)
        for (int v = seg_beg + lane; v < seg_end; v += 32) c += vec_ties<DT>(buf[r][v], v * E::kPerVec, n, sh.rs[r].kstar);
      c = warp_sum_u32(c);
      if (lane == 0) sh.w_tie[warp][r] = c;
    }
    __syncthreads();
    if (tid == 0)
      for (int r = 0; r < nrows; ++r) {
        uint32_t s = 0;
        for (int w = 0; w < kWarps; ++w) s += sh.w_tie[w][r];
        sh.x_tie[r] = s;
      }
    cluster.sync();
    for (int r = 0; r < nrows; ++r) {
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
  const RowStat rq = has_q ? sh.rs[1] : sh.rs[0];

  // ----------------------------------------------- MODE_PROBS: write rows
  if (a.mode == MODE_PROBS) {
    float* out = a.out_probs + static_cast<size_t>(unit) * V + lo;
    uint32_t run = warp_tie_base[0];
    for (int it = 0; it < seg_iters; ++it) {
      const int v = seg_beg + it * 32 + lane;
      const bool valid = v < seg_end;
      const uint4 x = valid ? buf[0][v] : make_uint4(0u, 0u, 0u, 0u);
      uint32_t base = 0;
      if (rp.partial) {
        const uint32_t c = valid ? vec_ties<DT>(x, v * E::kPerVec, n, rp.kstar) : 0u;
        const uint32_t incl = warp_incl_scan_u32(c);
        base = run + incl - c;
        run += __shfl_sync(kFull, incl, 31);
      }
      if (valid) {
        float w[8];
        draw_weights<DT>(x, x, v * E::kPerVec, n, false, rp, rp, cexp, cexp, base, base, w);
#pragma unroll
        for (int j = 0; j < E::kPerVec; ++j)
          if (v * E::kPerVec + j < n) out[v * E::kPerVec + j] = rp.bad ? 0.f : w[j];
      }
    }
    if (rp.bad && crank == 0 && tid == 0) set_status(a.status, SPEC_STATUS_BAD_ROW);
    cluster.sync();
    return;
  }

  // ------------------------------------- phase 3: accept test at x_pos
  const int kq = a.k;
  if (has_q) {
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
      // tie ranks of x inside this CTA (partial rows only)
      if (part_any) {
        for (int r = 0; r < 2; ++r) {
          uint32_t c = 0;
          if (sh.rs[r].partial)
            for (int t = tid; t < x - lo; t += kThreads)
              c += (E::key(E::bits_at(buf[r], t)) == sh.rs[r].kstar);
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

  // ------------------------- phase 4: residual (or bonus) inverse-CDF draw
  if (any_bad) {
    cluster.sync();
    if (crank == 0 && tid == 0) {
      a.recs[unit].drawn = -1;
      set_status(a.status, SPEC_STATUS_BAD_ROW);
      __threadfence();
      if (atomicAdd(a.tickets + b, 1u) == static_cast<uint32_t>(2 * kq)) sample_finalize(a, b);
    }
    return;
  }
  const float u_draw = a.uniforms[static_cast<size_t>(b) * (kq + 2) + (has_q ? kq + 1 : kq)];
  bool use_q = has_q;
  double S = 0.0, Pc = 0.0;
  int owner = -1;
  for (int attempt = 0; attempt < 2; ++attempt) {
    float s = 0.f;
    uint32_t runp = warp_tie_base[0], runq = warp_tie_base[1];
    for (int it = 0; it < seg_iters; ++it) {
      const int v = seg_beg + it * 32 + lane;
      const bool valid = v < seg_end;
      const uint4 xp = valid ? buf[0][v] : make_uint4(0u, 0u, 0u, 0u);
      const uint4 xq = (valid && use_q) ? buf[1][v] : make_uint4(0u, 0u, 0u, 0u);
      uint32_t bp = 0, bq = 0;
      if (part_any) {
        const int t0 = v * E::kPerVec;
        const uint32_t cp = (valid && rp.partial) ? vec_ties<DT>(xp, t0, n, rp.kstar) : 0u;
        const uint32_t cq = (valid && use_q && rq.partial) ? vec_ties<DT>(xq, t0, n, rq.kstar) : 0u;
        const uint32_t ip = warp_incl_scan_u32(cp), iq = warp_incl_scan_u32(cq);
        bp = runp + ip - cp;
        bq = runq + iq - cq;
        runp += __shfl_sync(kFull, ip, 31);
        runq += __shfl_sync(kFull, iq, 31);
      }
      if (valid) {
        float w[8];
        draw_weights<DT>(xp, xq, v * E::kPerVec, n, use_q, rp, rq, cexp, cexp, bp, bq, w);
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < E::kPerVec; ++j) ls += w[j];
        s += ls;
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
    cluster.sync();  // ------------------------------------------ sync 3
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
  cluster.sync();  // ------------------------------------------------- sync 4 (no DSMEM after this)

  if (owner == crank) {
    const double target = (double)u_draw * S - Pc;
    if (tid == 0) {
      double run = 0.0;
      int wsel = -1;
      double wbase = 0.0;
      int wlast = -1;
      double lbase = 0.0;
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
        const uint4 xq = (valid && use_q) ? buf[1][v] : make_uint4(0u, 0u, 0u, 0u);
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
          draw_weights<DT>(xp, xq, t0, n, use_q, rp, rq, cexp, cexp, bp, bq, w);
#pragma unroll
          for (int j = 0; j < E::kPerVec; ++j) {
            ls += w[j];
            if (w[j] > 0.f) lpos = t0 + j;
          }
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
