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
// How (one GPU, memory-bound).  Every row (the target and draft rows of
// each draft position (b, i), then the bonus target rows (b, k)) has a stream
// part and a tail part, run by one CTA each: as work items of one
// cooperative launch (every stream part, then every tail part; a tail part
// polls, bounded, for its row's stream part) or as two launches.
// The stream part reads its row from HBM once, 16-byte non-allocating loads
// by warp segments in index order:
//   - masses are taken on a power-of-two lattice: with c = log2(e) / T and
//     an integer k_t >= max(l) * c held per thread, mass(l) = 2^(l c - k_t)
//     (one packed f32x2 fma and one ex2 per element).  Raising k_t rescales
//     the running sum by an exact power of two, so the row sum
//     Z = sum 2^(l c - K) (K the CTA-wide k) carries no rescaling error;
//     2^(l c - K) / Z is the softmax of l / T.
//   - candidate vectors: a lane tags every 16-byte vector whose maximum is
//     within kTheta octaves of mass of the best maximum it knows (its own
//     running maximum, or the CTA's, exchanged at fixed stream steps).  A tag
//     is the vector's index in the warp segment and the bf16 pattern of its
//     maximum.  A lane list short of room drops the tags below its current
//     bound and, if still short, raises the lane's floor above its smallest
//     tag; each list is complete above max(bound, floor).
// It hands over a row header (maximum, lattice exponent, row sum, window
// bottom) and the tags at or above the window bottom.
// The tail part bounds the cut from the tagged maxima (vector maxima are
// tokens of the row, so the mass or count above a value is at least that of
// the maxima above it), gathers the tagged vectors at or above the bound in
// index order, counts their elements in a histogram of exact values and
// scans it for the cut, its tie count and the kept normaliser.  A row the
// candidates do not decide re-reads itself in windows of exact values from
// the maximum down, and past a few windows (flat rows crossing zero, 32-bit
// keys) by a bitwise search.  Each row publishes its state, its probability
// at the draft token and, for target rows, its vectors holding kept tokens.
// The last row of a sequence to finish (ticket, no spin-wait) tests
// u_i q_i(x_i) < p_i(x_i) at every position, takes the first rejection n,
// commits the accepted prefix and, when row n's kept vectors are listed,
// draws the token at n from max(0, p_n - q_n) (or from p_k when n = k) over
// them.  A draw over whole rows (no filter, or a row the candidates did not
// decide) is left to the draw kernel, which splits the rows into chunks.
// Only the first rejection is drawn: no residual is computed speculatively.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>

#include <algorithm>

#include "device_common.cuh"

namespace specv {

namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
using u64 = unsigned long long;

constexpr int kLaneTags = 32;                       // candidate vector tags per lane per row
constexpr int kBmapWords = 128;                     // gather bitmap words per warp per row (4096 vectors)
constexpr int kGather = kLaneTags * 32;             // gathered vectors per warp per row (in the lane tags' place)
constexpr int kSyncEvery = 4;                       // stream iterations between CTA maximum exchanges
constexpr float kTheta = 13.f;                      // octaves of mass kept as candidates
constexpr uint32_t kSlotMask = static_cast<uint32_t>(kWindow) - 1u;
// Histogram slot of a key (any kWindow consecutive keys take distinct
// slots): the low bits are mixed with bits 4.. so that the scan's lanes,
// which read keys 16 apart, fall in distinct shared-memory banks.
__device__ __forceinline__ uint32_t hslot(uint32_t key) { return (key & kSlotMask) ^ ((key >> 4) & 15u); }
constexpr int kGroups = kWindow / 4;                // aligned groups of four keys
constexpr int kScanWarps = 4;                       // warps that scan one row's histogram
constexpr int kVecCacheAt = 256;                    // gathered tags before, cached vectors after (words)
constexpr int kVecCache = (kGather - kVecCacheAt) / 4;  // cached gathered vectors per warp (192)

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
using RowStat = RowState;


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

// Row-wide values after the stream (the same for every thread).
struct RowG {
  float m;               // row maximum
  float K;               // lattice exponent
  uint32_t kmax;         // key of m
  uint32_t klo;          // lowest key of the scanned window
  DF z;                  // sum of masses 2^(l c - K)
  uint32_t c0;           // tokens above the window (keys > kmax)
  DF m0;                 // their mass
  int active;            // the row takes part in the current scan
};

struct Shm {
  float w_m[kWarps][2];
  int w_k[kWarps][2];
  float w_z[kWarps][2];
  uint32_t w_floor[kWarps][2]; // key above which a warp's tag list is complete
  uint32_t w_over[kWarps][2];  // a warp's gather overflowed
  float w_s[kWarps];
  float w_sp[kWarps];
  uint32_t w_u[kWarps][2];
  float x_m[2][kWarps][2];     // running maxima exchanged while streaming (double-buffered)
  uint32_t xbits[2];           // the draft token's value in the target and draft rows
  uint32_t s_C[2][kScanWarps];
  DF s_M[2][kScanWarps];
  RowG g[2];
  CutOut cutk[2];
  CutOut cut[2];
  int tie_warp[2];
  uint32_t tie_j[2];
  int tie_cut[2];
  int lead;                    // the warp that runs one-warp steps for this row
  RowStat rs[2];
  int draw_warp;
  float draw_base;
  int second;                  // this CTA is the last of its sequence (tail, draw kernels)
  int draw_chunk;              // the chunk holding the draw target, or -1
  int draw_useq;               // the draw weights are max(0, p - q)
  int draw_token;
  DF draw_target;              // the draw target within its chunk
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
  constexpr int kU = 4;  // loads in flight per thread
  uint32_t cnt = 0, kmin = 0xFFFFFFFFu;
  float mass = 0.f;
  for (int v0 = threadIdx.x; v0 < nvec; v0 += kU * kThreads) {
    uint4 xs[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = v0 + u * kThreads;
      xs[u] = v < nvec ? load_vec<DT>(row, v, V, aligned) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = v0 + u * kThreads;
#pragma unroll
      for (int j = 0; j < E::kPerVec; ++j) {
        if (v * E::kPerVec + j < V) {
          const uint32_t b = E::bits_of(xs[u], j);
          const uint32_t k = E::key(b);
          if (kind == PASS_COUNT_GE) cnt += (k >= kappa);
          else if (kind == PASS_COUNT_EQ) cnt += (k == kappa);
          else if (kind == PASS_MIN_GE) { if (k >= kappa) kmin = min(kmin, k); }
          else if (k > kappa) mass += lat_mass(E::value(b), rs.c, rs.K);
        }
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

// Warp w owns vectors [beg, end) of a row: consecutive vectors in index
// order (iteration, lane, element).
struct Seg {
  int beg, end, iters;
};
__device__ __forceinline__ int seg_vectors(int nvec) { return ((nvec + kWarps - 1) / kWarps + 31) / 32 * 32; }
__device__ __forceinline__ Seg warp_seg(int nvec, int warp) {
  const int vpw = seg_vectors(nvec);
  Seg s;
  s.beg = min(nvec, warp * vpw);
  s.end = min(nvec, s.beg + vpw);
  s.iters = (s.end - s.beg + 31) / 32;
  return s;
}

// Tag of a candidate vector: its index within the warp segment (high 16
// bits) and the bf16 pattern of its maximum (low 16 bits).
__device__ __forceinline__ uint32_t tag_make(uint32_t local, uint32_t key) { return (local << 16) | key; }
__device__ __forceinline__ uint32_t tag_local(uint32_t t) { return t >> 16; }
// (the tag keeps the maximum's bf16 pattern; its key orders the values)
__device__ __forceinline__ uint32_t tag_key(uint32_t t) { return Elt<DT_BF16>::key(t & 0xFFFFu); }

// Lane tag lists: every lane keeps the tags of the candidate vectors it
// streamed (stream order), kLaneTags per row; tag q of a lane sits at
// [row][warp][q][lane] (conflict-free).
__device__ __forceinline__ uint32_t lane_tags_purge(uint32_t* L, uint32_t n, uint32_t kthr) {
  uint32_t out = 0;
  for (uint32_t q = 0; q < n; ++q) {
    const uint32_t t = L[32 * q];
    if (tag_key(t) >= kthr) L[32 * (out++)] = t;
  }
  return out;
}
__device__ __forceinline__ uint32_t lane_tags_min_key(const uint32_t* L, uint32_t n) {
  uint32_t k = 0xFFFFFFFFu;
  for (uint32_t q = 0; q < n; ++q) k = min(k, tag_key(L[32 * q]));
  return k;
}

// The gathered vectors of one warp and row: its tags at or above the bound
// (index order); the vectors themselves are read from the row on demand.
struct GList {
  const uint32_t* tags;
  const unsigned char* row;
  const uint4* vc;  // the gathered vectors themselves (same order), or null: read from the row
};


// The cut of the row from a histogram of exact keys (slot key & (kWindow -
// 1), keys g.klo .. g.kmax), scanned by one warp from the top: lane l holds
// the 16 keys below 4 * (kmax >> 2) + 3 - 16 l, their counts and lattice
// masses summed, then one warp-wide prefix (count, double-float mass).
// Top-k: where the running count reaches top_k (sh.cutk); top-p (on the
// top-k set, if any): where the running mass reaches top_p * Z, a token being
// kept while the mass ranked before it is below the target (sh.cut).  The
// lane holding a crossing walks its 16 keys.  A cut below the window leaves
// found = 0.  The count and mass above the window (g.c0, g.m0) start the
// running sums; the window's own totals are left in sh.s_C[0][0], sh.s_M[0][0].
// With given_k the top-k cut in sh.cutk is taken as found earlier and only
// top-p is scanned.  Whole CTA (one barrier).
template <int DT, int NR>
__device__ __noinline__ void cut_scan(Shm& sh, const uint32_t* hist, float c, int top_k, float top_p,
                                      bool given_k = false) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool topk_on = top_k > 0, topp_on = top_p < 1.f;
  if (warp == sh.lead) {
    const RowG g = sh.g[0];
    CutOut ck = sh.cutk[0];
    if (!given_k) ck.found = 0;
    __syncwarp();
    if (lane == 0) {
      sh.cut[0].found = 0;
      if (!given_k) sh.cutk[0].found = 0;
    }
    __syncwarp();
    const uint32_t gtop = g.kmax >> 2;
    const uint32_t span = 4u * gtop + 3u;  // keys 0 .. span; lane l takes span - 16 l down to span - 16 l - 15
    const uint32_t top = span - 16u * static_cast<uint32_t>(lane);
    const bool live = g.active && span >= 16u * static_cast<uint32_t>(lane);
    uint32_t Cl = 0u;
    float Ml = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {  // (selects, no branches)
      const uint32_t key = top - static_cast<uint32_t>(j);
      const bool in = live && 16u * static_cast<uint32_t>(lane) + static_cast<uint32_t>(j) <= span &&
                      key <= g.kmax && key >= g.klo;
      const uint32_t n = in ? hist[hslot(key)] : 0u;
      const float ms = lat_mass(value_of_key<DT>(key), c, g.K);
      Cl += n;
      Ml += n ? static_cast<float>(n) * ms : 0.f;
    }
    const uint32_t Craw = warp_incl_scan_u32(Cl);
    const DF Mraw = warp_incl_scan_df(DF{Ml, 0.f});
    const uint32_t Cin = Craw + g.c0, Cex = Cin - Cl;
    const DF Min = df_add2(g.m0, Mraw);
    DF Mex = df_shfl_up(Min, 1);
    if (lane == 0) Mex = g.m0;
    if (lane == 31) {  // the window's own totals
      sh.s_C[0][0] = Craw;
      sh.s_M[0][0] = Mraw;
    }
    if (lane > 0 && lane < kScanWarps) {
      sh.s_C[0][lane] = 0u;
      sh.s_M[0][lane] = DF{0.f, 0.f};
    }
    // The crossing lane's 16 keys resolved by the warp: lane j < 16 takes
    // its key j (count, mass), then one warp prefix over them.
    auto lane_keys = [&](int xl, uint32_t& key, uint32_t& n, float& ms) {
      const uint32_t topx = span - 16u * static_cast<uint32_t>(xl);
      const uint32_t jj = static_cast<uint32_t>(lane);
      key = topx - jj;
      const bool in = lane < 16 && 16u * static_cast<uint32_t>(xl) + jj <= span && key <= g.kmax && key >= g.klo;
      n = in ? hist[hslot(key)] : 0u;
      ms = lat_mass(value_of_key<DT>(key), c, g.K);
    };
    if (topk_on && !given_k) {  // the value where the running count reaches top_k
      const uint32_t Kc = static_cast<uint32_t>(top_k);
      const unsigned bal = __ballot_sync(kFull, live && Cin >= Kc && Cex < Kc);
      if (bal) {  // (warp-uniform)
        const int xl = __ffs(bal) - 1;
        uint32_t key, n;
        float ms;
        lane_keys(xl, key, n, ms);
        const uint32_t run0 = __shfl_sync(kFull, Cex, xl);
        const DF mb0 = DF{__shfl_sync(kFull, Mex.hi, xl), __shfl_sync(kFull, Mex.lo, xl)};
        const uint32_t ci = warp_incl_scan_u32(n);
        const DF mi = warp_incl_scan_df(DF{n ? static_cast<float>(n) * ms : 0.f, 0.f});
        DF me = df_shfl_up(mi, 1);
        if (lane == 0) me = DF{0.f, 0.f};
        const uint32_t before = run0 + ci - n;
        const unsigned hit = __ballot_sync(kFull, n > 0u && before < Kc && before + n >= Kc);
        if (hit && lane == __ffs(hit) - 1) {
          ck.kstar = key;
          ck.keep = Kc - before;
          ck.total = n;
          ck.found = 1;
          ck.zkept = df_add(df_add2(mb0, me), static_cast<float>(Kc - before) * ms);
          sh.cutk[0] = ck;
          if (!topp_on) sh.cut[0] = ck;
        }
        const int src = hit ? __ffs(hit) - 1 : 0;
        ck.found = __shfl_sync(kFull, hit ? 1 : 0, src);
        ck.kstar = __shfl_sync(kFull, ck.kstar, src);
        ck.keep = __shfl_sync(kFull, ck.keep, src);
        ck.total = __shfl_sync(kFull, ck.total, src);
        ck.zkept = DF{__shfl_sync(kFull, ck.zkept.hi, src), __shfl_sync(kFull, ck.zkept.lo, src)};
      }
    }
    if (topp_on && (!topk_on || ck.found)) {
      const DF target = df_mul_f(topk_on ? ck.zkept : g.z, top_p);
      // the first lane whose running mass reaches the target (a window
      // holding less than the target leaves the cut unfound)
      const unsigned bal = __ballot_sync(kFull, live && !df_lt(Min, target));
      const int xl = bal ? __ffs(bal) - 1 : 0;
      const DF mb0 = DF{__shfl_sync(kFull, Mex.hi, xl), __shfl_sync(kFull, Mex.lo, xl)};
      if (bal && df_lt(mb0, target)) {  // (warp-uniform)
        uint32_t key, n;
        float ms;
        lane_keys(xl, key, n, ms);
        uint32_t ce = n;
        if (topk_on) ce = key < ck.kstar ? 0u : (key == ck.kstar ? ck.keep : ce);
        const DF mi = warp_incl_scan_df(DF{ce ? static_cast<float>(ce) * ms : 0.f, 0.f});
        DF me = df_shfl_up(mi, 1);
        if (lane == 0) me = DF{0.f, 0.f};
        const DF before = df_add2(mb0, me), after = df_add2(mb0, mi);
        const unsigned hit = __ballot_sync(kFull, ce > 0u && !df_lt(after, target));
        // (rounding may leave the crossing past these keys: then all of the last one)
        const unsigned pos = __ballot_sync(kFull, ce > 0u);
        const int jc = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
        if (jc >= 0 && lane == jc) {
          CutOut cp;
          uint32_t keep = ce;
          if (hit) {
            const float need = df_float(df_add(target, -before.hi)) - before.lo;
            keep = static_cast<uint32_t>(ceilf(need / ms));
            keep = max(1u, min(keep, ce));
          }
          cp.kstar = key;
          cp.keep = keep;
          cp.total = n;
          cp.found = 1;
          cp.zkept = df_add(before, static_cast<float>(keep) * ms);
          sh.cut[0] = cp;
        }
      }
    }
  }
  __syncthreads();
}

// Exact counts of the row's tokens with keys in [klo, khi] (klo .. klo +
// kWindow - 1, slot hslot(key)), by one re-read of the row with four loads
// in flight per thread.  Whole CTA.
template <int DT>
__device__ __noinline__ void window_pass(uint32_t* hist, const unsigned char* row, int V, bool aligned,
                                         uint32_t klo, uint32_t khi, uint32_t* priv) {
  using E = Elt<DT>;
  constexpr int kU = 4;
  const int nvec = (V + E::kPerVec - 1) / E::kPerVec;
  // each warp counts into its own copy when priv is given (fewer colliding
  // atomics on the common values), then the copies are summed
  uint32_t* const mine = priv ? priv + (threadIdx.x >> 5) * kWindow : hist;
  for (int t = threadIdx.x; t < kWindow; t += kThreads) hist[t] = 0u;
  if (priv)
    for (int t = threadIdx.x; t < kWarps * kWindow; t += kThreads) priv[t] = 0u;
  __syncthreads();
  for (int v0 = threadIdx.x; v0 < nvec; v0 += kU * kThreads) {
    uint4 x[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = v0 + u * kThreads;
      x[u] = v < nvec ? load_vec<DT>(row, v, V, aligned) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int t0 = (v0 + u * kThreads) * E::kPerVec;
#pragma unroll
      for (int j = 0; j < E::kPerVec; ++j) {
        const uint32_t k = E::key(E::bits_of(x[u], j));
        if (t0 + j < V && k >= klo && k <= khi) red_add_shared(smem_addr(mine + hslot(k)), 1u);
      }
    }
  }
  __syncthreads();
  if (priv) {
    for (int t = threadIdx.x; t < kWindow; t += kThreads) {
      uint32_t sum = 0u;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) sum += priv[w * kWindow + t];
      hist[t] = sum;
    }
    __syncthreads();
  }
}

constexpr int kSlowWindows = 8;  // windows of kWindow keys tried before the bitwise search

// The exact cut of a row that the candidate vectors do not decide: windows
// of kWindow consecutive keys from the row maximum down, each counted by a
// re-read of the row and scanned with the count and mass above it carried,
// until the window holding the cut.  Top-k first; top-p then scans the same
// windows on the top-k set.  A cut more than kSlowWindows windows down
// takes the bitwise search.  Whole CTA; sh.g[0] is left as it was.
template <int DT>
__device__ __noinline__ CutOut window_cut(Shm& sh, uint32_t* hist, const unsigned char* row, int V, bool aligned,
                                          int top_k, float top_p, const RowStat& rs, double zfull,
                                          uint32_t* priv) {
  // (32-bit keys are too fine for windows of kWindow keys)
  if (Elt<DT>::kKeyBits > 16) return search_cut<DT>(sh, row, V, aligned, top_k, top_p, rs, zfull);
  const bool topk_on = top_k > 0, topp_on = top_p < 1.f;
  const RowG g0 = sh.g[0];
  bool ok = true;
#pragma unroll 1
  for (int phase = 0; phase < 2 && ok; ++phase) {
    const bool kphase = phase == 0;
    if (kphase ? !topk_on : !topp_on) continue;
    uint32_t hi = g0.kmax, c0 = 0u;
    DF m0{0.f, 0.f};
    bool found = false;
#pragma unroll 1
    for (int w = 0; w < kSlowWindows && !found; ++w) {
      const uint32_t gt = hi >> 2;
      const uint32_t lo = gt >= static_cast<uint32_t>(kGroups - 1) ? 4u * (gt - static_cast<uint32_t>(kGroups - 1)) : 0u;
      window_pass<DT>(hist, row, V, aligned, lo, hi, priv);
      if (threadIdx.x == 0) {
        RowG g = g0;
        g.kmax = hi;
        g.klo = lo;
        g.c0 = c0;
        g.m0 = m0;
        g.active = 1;
        sh.g[0] = g;
      }
      __syncthreads();
      cut_scan<DT, 1>(sh, hist, rs.c, top_k, kphase ? 1.f : top_p, !kphase);
      found = (kphase ? sh.cutk[0].found : sh.cut[0].found) != 0;
      if (!found) {
#pragma unroll
        for (int q = 0; q < kScanWarps; ++q) {
          c0 += sh.s_C[0][q];
          m0 = df_add2(m0, sh.s_M[0][q]);
        }
        if (lo == 0u) break;
        hi = lo - 1u;
      }
      __syncthreads();
    }
    ok = found;
  }
  CutOut co = sh.cut[0];
  __syncthreads();
  if (threadIdx.x == 0) sh.g[0] = g0;
  __syncthreads();
  if (!ok) co = search_cut<DT>(sh, row, V, aligned, top_k, top_p, rs, zfull);
  return co;
}

// Tie cut of a row: tokens of value kstar are kept in index order, the
// first `keep` of them.  Every warp counts its tokens (in its gathered
// vectors, or in its segment of the row re-read), the warp holding token
// number `keep` (0-based) finds its row index.  Whole CTA.
template <int DT, bool FROM_LIST>
__device__ __noinline__ int tie_cut_of(Shm& sh, const GList& L, uint32_t len, const unsigned char* row, int V,
                                       bool aligned, uint32_t kstar, uint32_t keep) {
  using E = Elt<DT>;
  using H = Hot<DT>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = (V + E::kPerVec - 1) / E::kPerVec;
  const Seg sg = warp_seg(nvec, warp);
  const uint32_t thr = H::thr_pack(E::bits_of_key(kstar));
  const int rounds = FROM_LIST ? static_cast<int>((len + 31) / 32) : sg.iters;
  auto vec_at = [&](int it, uint4& x) -> int {
    if (FROM_LIST) {
      const uint32_t i = it * 32 + lane;
      if (i >= len) return -1;
      const int v = sg.beg + static_cast<int>(tag_local(L.tags[i]));
      x = L.vc ? L.vc[i] : load_vec<DT>(L.row, v, V, aligned);
      return v;
    }
    const int v = sg.beg + it * 32 + lane;
    if (v >= sg.end) return -1;
    x = load_vec<DT>(row, v, V, aligned);
    return v;
  };
  uint32_t c = 0;
  for (int it = 0; it < rounds; ++it) {
    uint4 x;
    const int v = vec_at(it, x);
    if (v >= 0) c += __popc(H::mask_eq(x, thr) & vmask<DT>(v, V));
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
    for (int it = 0; it < rounds; ++it) {
      uint4 x;
      const int v = vec_at(it, x);
      const uint32_t msk = v >= 0 ? (H::mask_eq(x, thr) & vmask<DT>(v, V)) : 0u;
      const uint32_t cc = __popc(msk);
      const uint32_t incl = warp_incl_scan_u32(cc);
      const uint32_t tot = __shfl_sync(kFull, incl, 31);
      if (jj < tot) {
        if (incl > jj && incl - cc <= jj) {
          uint32_t mm = msk;
          for (uint32_t q = jj - (incl - cc); q > 0; --q) mm &= mm - 1u;
          sh.tie_cut[0] = v * E::kPerVec + (__ffs(mm) - 1);
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
__device__ __noinline__ void write_probs(const unsigned char* row, int V, bool aligned, const RowStat& rp_in,
                                         float* out) {
  const RowStat rp = rp_in;
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

// Draw weights of the elements of one vector (row index v): max(0, p - q)
// (use_q) or p.  xq: the draft row's vector, or null when it holds no kept
// token of q.  Returns the sum; *ps gets the sum of p.
template <int DT>
__device__ __forceinline__ float vec_weights(const RowStat& rp, const RowStat& rq, const uint4& xp, const uint4* xq, int v,
                                             int V, bool use_q, float* w, float* ps) {
  using E = Elt<DT>;
  float s = 0.f, sp = 0.f;
  const uint32_t vm = vmask<DT>(v, V);
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = 0.f;
#pragma unroll
  for (int j = 0; j < E::kPerVec; ++j) {
    if ((vm >> j) & 1u) {
      const int t = v * E::kPerVec + j;
      const float pv = prob_of<DT>(rp, E::bits_of(xp, j), t);
      float wj = pv;
      if (use_q) {
        const float qv = (xq && pv > 0.f) ? prob_of<DT>(rq, E::bits_of(*xq, j), t) : 0.f;
        wj = fmaxf(pv - qv, 0.f);
      }
      w[j] = wj;
      s += wj;
      sp += pv;
    }
  }
  *ps = sp;
  return s;
}

}  // namespace

constexpr int ROLE_P = 0;      // target row of a draft position
constexpr int ROLE_Q = 1;      // draft row of a draft position
constexpr int ROLE_BONUS = 2;  // target row after the last draft
constexpr int ROLE_PROBS = 3;  // one row of spec_transform_probs

// The row of CTA `cta` in the stream and tail kernels: the target (even) and
// draft (odd) rows of every draft position, then the bonus target rows
// (MODE_PROBS: row cta).
struct RowRef {
  int role, b, pos;
  const unsigned char* row;
  bool aligned;
};
template <int DT>
__device__ __forceinline__ RowRef row_ref(const SampleArgs& a, int cta) {
  using E = Elt<DT>;
  const unsigned char* tgt = static_cast<const unsigned char*>(a.target);
  const size_t rb = static_cast<size_t>(a.V) * E::kBytes;
  RowRef r;
  if (a.mode == MODE_PROBS) {
    r.role = ROLE_PROBS;
    r.b = cta;
    r.pos = 0;
    r.row = tgt + static_cast<size_t>(cta) * rb;
    r.aligned = a.aligned_target != 0;
    return r;
  }
  const int k = a.k, npairs = a.B * k;
  if (cta < 2 * npairs) {
    const int pair = cta >> 1;
    r.role = (cta & 1) ? ROLE_Q : ROLE_P;
    r.b = pair / k;
    r.pos = pair % k;
    r.row = r.role == ROLE_P ? tgt + static_cast<size_t>(r.b * (k + 1) + r.pos) * rb
                             : static_cast<const unsigned char*>(a.draft) + static_cast<size_t>(pair) * rb;
    r.aligned = (r.role == ROLE_P ? a.aligned_target : a.aligned_draft) != 0;
  } else {
    r.role = ROLE_BONUS;
    r.b = cta - 2 * npairs;
    r.pos = k;
    r.row = tgt + static_cast<size_t>(r.b * (k + 1) + k) * rb;
    r.aligned = a.aligned_target != 0;
  }
  return r;
}

// -------------------------------------------------------------- the draw
// Entries [e0, e1) of a draw: row vector L[e] (index order, read past L1:
// written by another CTA of the same kernel) when L is given,
// else vector e itself; warp w takes the w-th of kWarps equal parts.
struct Part {
  int beg, end;
};
__device__ __forceinline__ Part warp_part(int e0, int e1, int warp) {
  const long long m = e1 - e0;
  Part p;
  p.beg = e0 + static_cast<int>(m * warp / kWarps);
  p.end = e0 + static_cast<int>(m * (warp + 1) / kWarps);
  return p;
}

// Per-warp sums of the draw weights over entries [e0, e1): max(0, p - q)
// (want_q) into sh.w_s and p into sh.w_sp.  Each lane sums its entries in
// order, four loads in flight; fixed-order warp sums.  Whole CTA.
template <int DT>
__device__ __noinline__ void range_sums(Shm& sh, const RowStat& rp_in, const RowStat& rq_in, const unsigned char* rowp,
                                        const unsigned char* rowq, bool ap, bool aq, int V, bool want_q,
                                        const uint32_t* L, int e0, int e1) {
  const RowStat rp = rp_in, rq = rq_in;  // (register copies: no reloads through the references)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Part pt = warp_part(e0, e1, warp);
  constexpr int kU = 4;
  float s = 0.f, sp = 0.f;
  for (int e = pt.beg + lane; e < pt.end; e += 32 * kU) {
    uint4 xp[kU], xq[kU];
    int vv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int ee = e + 32 * u;
      vv[u] = ee < pt.end ? (L ? static_cast<int>(__ldcg(L + ee)) : ee) : -1;
      if (vv[u] >= 0) {
        xp[u] = load_vec<DT>(rowp, vv[u], V, ap);
        xq[u] = want_q ? load_vec<DT>(rowq, vv[u], V, aq) : xp[u];
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (vv[u] >= 0) {
        float w[8], ps;
        s += vec_weights<DT>(rp, rq, xp[u], &xq[u], vv[u], V, want_q, w, &ps);
        sp += ps;
      }
    }
  }
  s = warp_sum_f32(s);
  sp = warp_sum_f32(sp);
  if (lane == 0) {
    sh.w_s[warp] = s;
    sh.w_sp[warp] = sp;
  }
  __syncthreads();
}

// The token at cumulative weight tw (relative to e0) over entries [e0, e1),
// given their per-warp sums in sh (range_sums): the warp holding tw walks its
// part in index order.  -1 when the range has no weight.  Whole CTA; every
// thread gets the token.
template <int DT>
__device__ __noinline__ int range_walk(Shm& sh, const RowStat& rp_in, const RowStat& rq_in, const unsigned char* rowp,
                                       const unsigned char* rowq, bool ap, bool aq, int V, bool use_q, DF tw_in,
                                       const uint32_t* L, int e0, int e1) {
  const RowStat rp = rp_in, rq = rq_in;  // (register copies: no reloads through the references)
  using E = Elt<DT>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    const float* ws = use_q ? sh.w_s : sh.w_sp;
    DF run{0.f, 0.f}, base{0.f, 0.f}, lbase{0.f, 0.f};
    int wsel = -1, wlast = -1;
    for (int w = 0; w < kWarps; ++w) {
      const float sw = ws[w];
      const DF nxt = df_add(run, sw);
      if (sw > 0.f) { wlast = w; lbase = run; }
      if (wsel < 0 && sw > 0.f && df_lt(tw_in, nxt)) { wsel = w; base = run; }
      run = nxt;
    }
    if (wsel < 0) { wsel = wlast; base = lbase; }
    sh.draw_warp = wsel;
    sh.draw_base = df_float(df_add2(tw_in, df_neg(base)));
    sh.draw_token = -1;
  }
  __syncthreads();
  if (warp == sh.draw_warp) {
    const Part pt = warp_part(e0, e1, warp);
    const float tw = sh.draw_base;
    const int rounds = (pt.end - pt.beg + 31) / 32;
    float run = 0.f;
    int token = -1, last_pos = -1;
    constexpr int kR = 2;  // rounds whose vectors are read together
    for (int it0 = 0; it0 < rounds && token < 0; it0 += kR) {
    int vr[kR];
    uint4 xpr[kR], xqr[kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      const int e = pt.beg + (it0 + r) * 32 + lane;
      vr[r] = (it0 + r < rounds && e < pt.end) ? (L ? static_cast<int>(__ldcg(L + e)) : e) : -1;
    }
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      if (vr[r] >= 0) {
        xpr[r] = load_vec<DT>(rowp, vr[r], V, ap);
        xqr[r] = use_q ? load_vec<DT>(rowq, vr[r], V, aq) : xpr[r];
      }
    }
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      if (it0 + r >= rounds || token >= 0) break;
      const int v = vr[r];
      float w[8], ps;
      float ls = 0.f;
      int lpos = -1;
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = 0.f;
      if (v >= 0) {
        const uint4 xp = xpr[r];
        const uint4 xq = xqr[r];
        ls = vec_weights<DT>(rp, rq, xp, &xq, v, V, use_q, w, &ps);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (w[j] > 0.f) lpos = v * E::kPerVec + j;
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
            if (w[j] > 0.f) lastj = v * E::kPerVec + j;
            cum += w[j];
            if (tok < 0 && w[j] > 0.f && cum > tw) tok = v * E::kPerVec + j;
          }
          if (tok < 0) tok = lastj;
        }
        token = __shfl_sync(kFull, tok, l);
      }
      run += __shfl_sync(kFull, incl, 31);
    }
    }
    if (token < 0) token = last_pos;  // only reachable through rounding
    if (lane == 0) sh.draw_token = token;
  }
  __syncthreads();
  return sh.draw_token;
}


// The draw over a target row's listed kept vectors (N <= kPubList entries):
// every thread reads its entries and their vector pairs at once and keeps
// each entry's weight sums (max(0, p - q), and p) in shared memory; per-warp
// sums in the order of range_sums; the warp holding u * S finds the entry
// from the kept sums and reads only that entry's vectors again to pick the
// token (as range_walk).  idx: kPubList words, ew: 2 * kPubList floats of
// shared memory.  Whole CTA; every thread gets the token.
template <int DT>
__device__ __noinline__ int draw_listed(Shm& sh, const RowStat& rp_in, const RowStat& rq_in, const unsigned char* rowp,
                                        const unsigned char* rowq, bool ap, bool aq, int V, bool want_q,
                                        const uint32_t* Lg, int N, float u, uint32_t* idx, float* ew) {
  const RowStat rp = rp_in, rq = rq_in;  // (register copies: no reloads through the references)
  using E = Elt<DT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kPer = kPubList / kThreads;  // entries per thread, two pairs of rows' vectors in flight
#pragma unroll 1
  for (int jb = 0; jb < kPer && tid + kThreads * jb < N; jb += 2) {
    int vv[2];
    uint4 xp[2], xq[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int e = tid + kThreads * (jb + j);
      vv[j] = e < N ? static_cast<int>(__ldcg(Lg + e)) : -1;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (vv[j] >= 0) {
        xp[j] = load_vec<DT>(rowp, vv[j], V, ap);
        xq[j] = want_q ? load_vec<DT>(rowq, vv[j], V, aq) : xp[j];
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (vv[j] >= 0) {
        const int e = tid + kThreads * (jb + j);
        float w[8], ps;
        ew[2 * e] = vec_weights<DT>(rp, rq, xp[j], &xq[j], vv[j], V, want_q, w, &ps);
        ew[2 * e + 1] = ps;
        idx[e] = static_cast<uint32_t>(vv[j]);
      }
    }
  }
  __syncthreads();
  const Part pt = warp_part(0, N, warp);
  {
    float s = 0.f, sp = 0.f;
    for (int e = pt.beg + lane; e < pt.end; e += 32) {
      s += ew[2 * e];
      sp += ew[2 * e + 1];
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
    DF tr{0.f, 0.f}, tp{0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      tr = df_add(tr, sh.w_s[w]);
      tp = df_add(tp, sh.w_sp[w]);
    }
    const bool use_q = want_q && tr.hi > 0.f;  // a residual with no mass: draw from p
    const DF target = df_mul_f(use_q ? tr : tp, u);
    const float* ws = use_q ? sh.w_s : sh.w_sp;
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
    sh.draw_useq = use_q ? 1 : 0;
    sh.draw_warp = wsel;
    sh.draw_base = df_float(df_add2(target, df_neg(base)));
    sh.draw_token = -1;
  }
  __syncthreads();
  if (warp == sh.draw_warp) {
    const bool use_q = sh.draw_useq != 0;
    const float tw = sh.draw_base;
    const int o = use_q ? 0 : 1;
    float run = 0.f, cum0 = 0.f;
    int ecross = -1, elast = -1;
    for (int e0 = pt.beg; e0 < pt.end && ecross < 0; e0 += 32) {
      const int e = e0 + lane;
      const float ls = e < pt.end ? ew[2 * e + o] : 0.f;
      const float incl = warp_incl_scan(ls);
      const unsigned ball = __ballot_sync(kFull, ls > 0.f && run + incl > tw);
      const unsigned pos = __ballot_sync(kFull, ls > 0.f);
      if (pos) elast = e0 + 31 - __clz(pos);
      if (ball) {
        const int l = __ffs(ball) - 1;
        ecross = e0 + l;
        cum0 = __shfl_sync(kFull, run + (incl - ls), l);
      }
      run += __shfl_sync(kFull, incl, 31);
    }
    // the entry holding the target (or, only through rounding, the last
    // entry with weight): its elements walked in order
    const int ee = ecross >= 0 ? ecross : elast;
    if (lane == 0 && ee >= 0) {
      const int v = static_cast<int>(idx[ee]);
      const uint4 xp = load_vec<DT>(rowp, v, V, ap);
      const uint4 xq = use_q ? load_vec<DT>(rowq, v, V, aq) : xp;
      float w[8], ps;
      vec_weights<DT>(rp, rq, xp, &xq, v, V, use_q, w, &ps);
      int tok = -1, lastj = -1;
      float cum = cum0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (w[j] > 0.f) lastj = v * E::kPerVec + j;
        cum += w[j];
        if (ecross >= 0 && tok < 0 && w[j] > 0.f && cum > tw) tok = v * E::kPerVec + j;
      }
      sh.draw_token = tok >= 0 ? tok : lastj;
    }
  }
  __syncthreads();
  return sh.draw_token;
}

// A row's published state, read past L1 (written by another CTA).
__device__ __forceinline__ RowStat ldcg_rowstat(const RowStat* p) {
  RowStat r;
  const uint32_t* s = reinterpret_cast<const uint32_t*>(p);
  uint32_t* d = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int i = 0; i < static_cast<int>(sizeof(RowStat) / 4); ++i) d[i] = __ldcg(s + i);
  return r;
}

// The records of sequence b's rows (pubs) zeroed for the next call, whatever
// its shape.  Whole CTA; every read of them is done.
// nl_pre: the rows' list lengths already in shared memory, or null.
__device__ __noinline__ void clear_sequence_pubs(const SampleArgs& a, int b, const uint32_t* nl_pre) {
  __shared__ uint32_t s_nl[2 * kMaxK + 1];
  const int k = a.k, nrows = 2 * k + 1, tid = threadIdx.x;
  auto row_pub = [&](int r) { return r < 2 * k ? a.pubs + 2 * static_cast<size_t>(b) * k + r
                                                 : a.pubs + 2 * static_cast<size_t>(a.B) * k + b; };
  __syncthreads();
  if (!nl_pre && tid < nrows) s_nl[tid] = __ldcg(&row_pub(tid)->nlist);
  __syncthreads();
  const uint32_t* const nls = nl_pre ? nl_pre : s_nl;
  for (int r = 0; r < nrows; ++r) {
    const uint32_t nl = nls[r];
    if (nl != kPubReread)
      for (uint32_t i = tid; i < nl && i < static_cast<uint32_t>(kPubList); i += kThreads) row_pub(r)->list[i] = 0u;
  }
  constexpr int kHdrWords = static_cast<int>(offsetof(RowPub, list) / 4);
  for (int i = tid; i < nrows * kHdrWords; i += kThreads)
    reinterpret_cast<uint32_t*>(row_pub(i / kHdrWords))[i % kHdrWords] = 0u;
}

constexpr uint32_t kDrawnInTail = 0x80000000u;  // draw ticket flag: the tail kernel drew the token

// ---------------------------------------------------------- stream kernel
// One CTA per row: stream it once (lattice masses, maximum, candidate tags),
// then hand over the row header and the tags at or above klo.
template <int DT>
__device__ __forceinline__ void stream_row(const SampleArgs& a, Shm& sh, uint32_t* dsm, const int cta) {
  using E = Elt<DT>;
  using H = Hot<DT>;
  uint32_t* const ltags = dsm;  // lane tags [kWarps][kLaneTags][32]
  const RowRef rr = row_ref<DT>(a, cta);
  const int role = rr.role, b = rr.b, pos = rr.pos;
  const unsigned char* const row = rr.row;
  const bool aligned = rr.aligned;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;
  const float T = a.temperature_per_seq ? a.temperature_per_seq[b] : a.temperature;
  const bool bad_t = !(T > 0.f) || isinf(T);
  const float c = kLog2e / T;
  const u64 c2 = pkf(c, c);
  const int nvec = (V + E::kPerVec - 1) / E::kPerVec;
  const Seg sg = warp_seg(nvec, warp);
  const bool filt = a.top_k > 0 || a.top_p < 1.f;
  const int kq = a.k;
  const bool paired = role == ROLE_P || role == ROLE_Q;
  const int xtok = paired ? a.tokens[static_cast<size_t>(b) * kq + pos] : -1;
  // candidate tags: bf16 rows with a cut, segments short enough to index
  const bool use_lists = DT == DT_BF16 && filt && !bad_t && seg_vectors(nvec) <= kBmapWords * 32;
  const float dtheta = kTheta / c;  // kTheta octaves of mass, in logit units
  uint32_t* const myl = ltags + warp * kLaneTags * 32 + lane;

  if (tid == 0) sh.xbits[0] = 0u;
  __syncthreads();

  // --------------------------------------------------- phase 1: stream
  float mt = -INFINITY;     // thread maximum
  int kt = -(1 << 30);      // thread lattice exponent
  u64 acc0 = 0ull, acc1 = 0ull;  // thread sums of 2^(l c - kt)
  float mw = -INFINITY;     // CTA maximum of the last exchange
  uint32_t cnt = 0u;        // lane tag list length
  uint32_t lfl = 0u;        // lane floor: the lane list is complete above it
  float lflv = -INFINITY;   // its value
  float lthr = -3.0e38f;    // lane bound: kTheta octaves below mw, at least the lane floor
                            // (finite: the -inf padding past a segment is never tagged)
  int sync_no = 0;
  // every warp runs the same number of iterations (the CTA barriers below)
  const int iters_all = seg_vectors(nvec) / 32;
  // whole 16-byte vectors: every vector below the segment end is full
  const bool whole = aligned && (V % E::kPerVec) == 0;
  for (int it = 0; it < iters_all; it += 4) {
    uint4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = sg.beg + (it + u) * 32 + lane;
      x[u] = make_uint4(H::kPad, H::kPad, H::kPad, H::kPad);
      if (v < sg.end) x[u] = whole ? ldg_stream(row + 16 * static_cast<size_t>(v)) : load_vec<DT>(row, v, V, aligned);
    }
    // the four vectors' maxima: one lattice-exponent check and one bound
    // update per four vectors
    float vmx[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) vmx[u] = H::vmax(x[u]);
    const float gm = max_nan(max_nan(vmx[0], vmx[1]), max_nan(vmx[2], vmx[3]));
    {
      const float L = gm * c;
      if (L > static_cast<float>(kt) && L < 1073741824.f) {  // raise the lattice exponent (rare)
        const int knew = static_cast<int>(ceilf(L));
        const float s = exp2i(kt - knew);
        acc0 = mul2(acc0, pkf(s, s));
        acc1 = mul2(acc1, pkf(s, s));
        kt = knew;
      }
    }
    const float nk = -static_cast<float>(kt);
    const u64 nk2 = pkf(nk, nk);
    mt = max_nan(mt, gm);
    // lane bound lthr: kTheta octaves below the larger of this lane's running
    // maximum and the CTA maximum of the last exchange (both at most the row
    // maximum), never below the lane floor
    lthr = fmaxf(lthr, gm - dtheta);
    if (use_lists && cnt > static_cast<uint32_t>(kLaneTags - 4)) {
      // (rare) room for this group's four candidates: drop the tags below the
      // bound, then while still short of room raise the lane's floor above its
      // smallest tag; the list stays complete above max(bound, floor)
      cnt = lane_tags_purge(myl, cnt, E::key(bits_round_down<DT>(lthr)));
      while (cnt > static_cast<uint32_t>(kLaneTags - 4)) {
        lfl = lane_tags_min_key(myl, cnt) + 1u;
        lflv = value_of_key<DT>(lfl);
        cnt = lane_tags_purge(myl, cnt, lfl);
      }
      lthr = fmaxf(lthr, lflv);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = sg.beg + (it + u) * 32 + lane;
      H::mass_vec(x[u], c2, nk2, acc0, acc1);
      // a candidate: one predicated store, no branch
      const bool take = use_lists && vmx[u] >= lthr;
      if (take) myl[32 * cnt] = (static_cast<uint32_t>(v - sg.beg) << 16) | (__float_as_uint(vmx[u]) >> 16);
      cnt += take ? 1u : 0u;
    }
    const int li = it >> 2;  // loop iteration
    if (use_lists && (li < kSyncEvery ? (li & (li + 1)) == 0 : (li % kSyncEvery) == kSyncEvery - 1)) {
      // share the running maxima across the CTA (fixed points, denser at the
      // start where they rise fastest: deterministic)
      const int slot = (sync_no++) & 1;
      const float wm = warp_max_nan(mt);
      if (lane == 0) sh.x_m[slot][warp][0] = fmaxf(mw, wm);
      __syncthreads();
      float mm = mw;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, sh.x_m[slot][w][0]);
      if (mm > mw) {
        mw = mm;
        lthr = fmaxf(lthr, mw - dtheta);
      }
    }
  }

  // the row's value at the draft token
  if (tid == 0 && xtok >= 0 && xtok < V) sh.xbits[0] = E::bits_at(row, xtok);

  // ------------------------------------------ phase 2: row maximum and sum
  {
    float s0, s1, s2, s3;
    upk(acc0, s0, s1);
    upk(acc1, s2, s3);
    float zt = (s0 + s1) + (s2 + s3);
    const int kw = warp_max_i32(kt);
    zt *= exp2i(kt - kw);
    zt = warp_sum_f32(zt);
    const float mx = warp_max_nan(mt);
    const uint32_t fl = warp_max_u32(lfl);
    if (lane == 0) {
      sh.w_m[warp][0] = mx;
      sh.w_k[warp][0] = kw;
      sh.w_z[warp][0] = zt;
      sh.w_floor[warp][0] = fl;
      sh.w_over[warp][0] = 0u;
    }
  }
  __syncthreads();
  if (tid == 0) {
    float mx = -INFINITY;
    int kk = -(1 << 30);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      mx = max_nan(mx, sh.w_m[w][0]);
      kk = max(kk, sh.w_k[w][0]);
    }
    DF z{0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kWarps; ++w) z = df_add(z, sh.w_z[w][0] * exp2i(sh.w_k[w][0] - kk));
    RowG g;
    g.m = mx;
    g.K = static_cast<float>(kk);
    g.kmax = key_of_float<DT>(mx);
    g.z = z;
    g.c0 = 0u;
    g.m0 = DF{0.f, 0.f};
    // every vector whose maximum reaches klo is tagged
    const float tv = mx - dtheta;
    uint32_t kl = tv > -3.0e38f ? E::key(bits_round_up<DT>(tv)) : 0u;
    const uint32_t gtop = g.kmax >> 2;
    if (gtop >= static_cast<uint32_t>(kGroups - 1)) kl = max(kl, 4u * (gtop - static_cast<uint32_t>(kGroups - 1)));
#pragma unroll
    for (int w = 0; w < kWarps; ++w) kl = max(kl, sh.w_floor[w][0]);
    g.klo = kl;
    g.active = use_lists ? 1 : 0;
    sh.g[0] = g;
  }
  __syncthreads();
  // the lattice exponent must stay an int: |max| log2(e) / T < 2^30
  const bool bad = bad_t || !isfinite(sh.g[0].m) || !(fabsf(sh.g[0].m * c) < 1073741824.f);

  // ------------- hand over: the row header and its tags at or above klo
  {
    const bool lists = use_lists && !bad;
    const uint32_t kl = sh.g[0].klo;
    uint32_t mine = 0u;
    if (lists)
      for (uint32_t q = 0; q < cnt; ++q) mine += tag_key(myl[32 * q]) >= kl ? 1u : 0u;
    const uint32_t incl = warp_incl_scan_u32(mine);
    if (lists) {
      uint32_t* dst = a.tags + static_cast<size_t>(cta) * kRowTags + warp * kTagsPerWarp;
      uint32_t o = incl - mine;  // (at most kLaneTags * 32 = kTagsPerWarp in all)
      for (uint32_t q = 0; q < cnt; ++q) {
        const uint32_t t = myl[32 * q];
        if (tag_key(t) >= kl) dst[o++] = t;
      }
    }
    if (lane == 31) sh.w_u[warp][0] = lists ? incl : 0u;
  }
  __syncthreads();
  if (tid == 0) {
    const RowG g = sh.g[0];
    RowHdr h;
    h.m = g.m;
    h.K = g.K;
    h.zhi = g.z.hi;
    h.zlo = g.z.lo;
    h.kmax = g.kmax;
    h.klo = g.klo;
    h.xbits = sh.xbits[0];
    h.bad = bad ? 1 : 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) h.ntags[w] = sh.w_u[w][0];
    a.hdrs[cta] = h;
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 4) stream_kernel(const SampleArgs a) {
  __shared__ Shm sh;
  extern __shared__ __align__(16) uint32_t dsm[];
  stream_row<DT>(a, sh, dsm, static_cast<int>(blockIdx.x));
}

// ------------------------------------------------------------ tail kernel
// One CTA per row, after the stream kernel: the kept set of the row from its
// header and tags (or by re-reading the row), published with its probability
// at the draft token and, for target rows, its kept vectors.  The last row
// of a sequence to finish applies the first-rejection rule.
// timed_out: the row's header never arrived (fused kernel): the row is
// published as bad without reading it.
template <int DT>
__device__ __forceinline__ void tail_row(const SampleArgs& a, Shm& sh, uint32_t* dsm, const int cta,
                                         const bool timed_out) {
  using E = Elt<DT>;
  using H = Hot<DT>;
  // dynamic shared memory: tags [kWarps][kTagsPerWarp] (then the gathered
  // tags in their place), histogram [kWindow], gather bitmaps
  // [kWarps][kBmapWords]
  uint32_t* const ltags = dsm;
  uint32_t* const hist = ltags + kRowTags;
  uint32_t* const bmap = hist + kWindow;
  const RowRef rr = row_ref<DT>(a, cta);
  const int role = rr.role, b = rr.b, pos = rr.pos;
  const unsigned char* const row = rr.row;
  const bool aligned = rr.aligned;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;
  const float T = a.temperature_per_seq ? a.temperature_per_seq[b] : a.temperature;
  const bool bad_t = !(T > 0.f) || isinf(T);
  const float c = kLog2e / T;
  const int nvec = (V + E::kPerVec - 1) / E::kPerVec;
  const Seg sg = warp_seg(nvec, warp);
  const bool topk_on = a.top_k > 0;
  const bool topp_on = a.top_p < 1.f;
  const bool filt = topk_on || topp_on;
  const int kq = a.k;
  const bool paired = role == ROLE_P || role == ROLE_Q;
  const int xtok = paired ? a.tokens[static_cast<size_t>(b) * kq + pos] : -1;
  const bool use_lists = DT == DT_BF16 && filt && !bad_t && seg_vectors(nvec) <= kBmapWords * 32;
  // a warp's tags, then its gathered vectors (index order)
  uint32_t* const wg = ltags + warp * kGather;
  uint32_t* const wb = bmap + warp * kBmapWords;
  GList gl;
  gl.tags = wg;
  gl.row = row;
  gl.vc = nullptr;
  // gathered vectors cached after the first kVecCacheAt words of the warp's region
  uint4* const vc = reinterpret_cast<uint4*>(wg + kVecCacheAt);

  // The header and the first tags are read together (the tag area beyond a
  // warp's count holds zeros), so one memory round trip covers most rows.
  // (read past L1: written by another CTA when the kernels are fused)
  const RowHdr* const hp = a.hdrs + cta;
  uint32_t* const src = a.tags + static_cast<size_t>(cta) * kRowTags + warp * kTagsPerWarp;
  constexpr int kSpec = 8;  // tags per lane read ahead of the count
  uint32_t t8[kSpec];
  if (use_lists && !timed_out) {
#pragma unroll
    for (int u = 0; u < kSpec; ++u) t8[u] = __ldcg(src + 32 * u + lane);
  }
  const bool bad = timed_out || __ldcg(&hp->bad) != 0;
  const uint32_t ntag = use_lists && !bad ? __ldcg(&hp->ntags[warp]) : 0u;
  if (tid == 0) {
    RowG g;
    g.m = timed_out ? 0.f : __ldcg(&hp->m);
    g.K = timed_out ? 0.f : __ldcg(&hp->K);
    g.kmax = timed_out ? 0u : __ldcg(&hp->kmax);
    g.klo = timed_out ? 0u : __ldcg(&hp->klo);
    g.z = timed_out ? DF{1.f, 0.f} : DF{__ldcg(&hp->zhi), __ldcg(&hp->zlo)};
    g.c0 = 0u;
    g.m0 = DF{0.f, 0.f};
    g.active = use_lists ? 1 : 0;
    sh.g[0] = g;
    sh.xbits[0] = timed_out ? 0u : __ldcg(&hp->xbits);
    // one-warp steps of co-resident CTAs spread over the SM's schedulers
    // (warp w issues from scheduler w % 4): a hashed warp per row
    sh.lead = static_cast<int>((static_cast<uint32_t>(cta) * 2654435761u) >> 29);
  }
  if (filt)
    for (int t = tid; t < kWindow; t += kThreads) hist[t] = 0u;
  {  // (the handed-over tags and header are left zeroed for the next call)
#pragma unroll
    for (int u = 0; u < kSpec; ++u) {
      const uint32_t i = 32 * u + lane;
      if (i < ntag) {
        wg[i] = t8[u];
        src[i] = 0u;
      }
    }
    for (uint32_t i0 = 32 * kSpec; i0 < ntag; i0 += 32 * 8) {  // the rest, eight loads in flight per lane
      uint32_t r8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t i = i0 + 32 * u + lane;
        r8[u] = i < ntag ? __ldcg(src + i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t i = i0 + 32 * u + lane;
        if (i < ntag) {
          wg[i] = r8[u];
          src[i] = 0u;
        }
      }
    }
  }
  __syncthreads();
  if (tid < static_cast<int>(sizeof(RowHdr) / 4)) reinterpret_cast<uint32_t*>(a.hdrs + cta)[tid] = 0u;

  // ---------- phase 3: a bound on the cut from the tagged vector maxima
  // The tags hold every vector whose maximum reaches klo.  Vector maxima
  // are tokens of the row, so the mass (or count) of the row above a value is
  // at least that of the maxima above it: where the maxima reach the top-p
  // target (or top_k), the row's cut lies at or above.
  int ngat = 0;
  bool fast = false;
  if (use_lists && !bad) {
    {
      const uint32_t kl = sh.g[0].klo;
      for (uint32_t i = lane; i < ntag; i += 32) {
        const uint32_t k = tag_key(wg[i]);
        if (k >= kl) red_add_shared(smem_addr(hist + hslot(k)), 1u);
      }
    }
    __syncthreads();
    cut_scan<DT, 1>(sh, hist, c, a.top_k, a.top_p);
    // bound (top-k: its own cut; top-p alone: the maxima's crossing)
    const CutOut bo = topk_on ? sh.cutk[0] : sh.cut[0];
    fast = bo.found != 0;
    const uint32_t tau = bo.kstar;
    __syncthreads();
    for (int t = tid; t < kWindow; t += kThreads) hist[t] = 0u;
    // the gathered vectors: the warp's tags at or above the bound, marked in
    // its bitmap and read back in index order (in the tags' place)
    if (fast) {
      const int nwords = seg_vectors(nvec) / 32;
      for (int w2 = lane; w2 < nwords; w2 += 32) wb[w2] = 0u;
      __syncwarp();
      for (uint32_t i = lane; i < ntag; i += 32) {
        const uint32_t t = wg[i];
        if (tag_key(t) >= tau) atomicOr(&wb[tag_local(t) >> 5], 1u << (tag_local(t) & 31u));
      }
      __syncwarp();
      uint32_t base = 0u;
      for (int w0 = 0; w0 < nwords; w0 += 32) {
        const int w2 = w0 + lane;
        const uint32_t bits = w2 < nwords ? wb[w2] : 0u;
        const uint32_t cb = __popc(bits);
        const uint32_t incl = warp_incl_scan_u32(cb);
        uint32_t o = base + incl - cb;
        uint32_t bb = bits;
        while (bb) {
          const uint32_t j = __ffs(bb) - 1u;
          bb &= bb - 1u;
          if (o < static_cast<uint32_t>(kGather)) wg[o] = tag_make(static_cast<uint32_t>(w2) * 32u + j, 0u);
          ++o;
        }
        base += __shfl_sync(kFull, incl, 31);
      }
      ngat = static_cast<int>(min(base, static_cast<uint32_t>(kGather)));
      if (lane == 0) sh.w_over[warp][0] = base > static_cast<uint32_t>(kGather) ? 1u : 0u;
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kWarps; ++w) fast = fast && sh.w_over[w][0] == 0u;
    // exact histogram of the gathered elements at or above the bound
    if (fast) {
      const uint32_t thr = H::thr_pack(E::bits_of_key(tau));
      const bool cache = ngat <= kVecCache;
      for (int i = lane; i < ngat; i += 32) {
        const int v = sg.beg + static_cast<int>(tag_local(wg[i]));
        const uint4 x = load_vec<DT>(row, v, V, aligned);
        if (cache) vc[i] = x;
        wg[i] = tag_make(tag_local(wg[i]), __float_as_uint(H::vmax(x)) >> 16);  // keep its maximum
        uint32_t msk = H::mask_ge(x, thr) & vmask<DT>(v, V);
        while (msk) {
          const int j = __ffs(msk) - 1;
          msk &= msk - 1u;
          red_add_shared(smem_addr(hist + hslot(E::key(E::bits_of(x, j)))), 1u);
        }
      }
    }
    if (tid == 0) {
      sh.g[0].klo = tau;
      sh.g[0].active = fast ? 1 : 0;
    }
    __syncthreads();
    cut_scan<DT, 1>(sh, hist, c, a.top_k, a.top_p);
    fast = fast && sh.cut[0].found != 0;
    if (fast && ngat <= kVecCache) gl.vc = vc;
  }


  // ------------------------------------------ phase 4: kept set of the row
  RowStat rs;
  {
    const RowG g = sh.g[0];
    rs.c = c;
    rs.K = g.K;
    rs.m = g.m;
    rs.kmax = g.kmax;
    rs.bad = bad ? 1 : 0;
    rs.all_kept = filt ? 0 : 1;
    rs.covered = fast ? 1 : 0;
    rs.kstar = 0u;
    rs.tie_cut = V;
    float zk = df_float(g.z);
    if (filt && !bad) {
      const CutOut co = fast ? sh.cut[0] : window_cut<DT>(sh, hist, row, V, aligned, a.top_k, a.top_p, rs, df_double(g.z),
                                                          use_lists ? ltags : nullptr);
      rs.kstar = co.kstar;
      zk = df_float(co.zkept);
      if (co.keep < co.total)
        rs.tie_cut = fast ? tie_cut_of<DT, true>(sh, gl, static_cast<uint32_t>(ngat), row, V, aligned, co.kstar, co.keep)
                          : tie_cut_of<DT, false>(sh, gl, 0u, row, V, aligned, co.kstar, co.keep);
    }
    rs.zkept = zk;
    rs.inv_z = 1.f / zk;
  }


  if (role == ROLE_PROBS) {
    float* out = a.out_probs + static_cast<size_t>(cta) * V;
    if (bad) {
      for (int t = tid; t < V; t += kThreads) out[t] = 0.f;
      if (tid == 0) set_status(a.status, SPEC_STATUS_BAD_ROW);
    } else {
      write_probs<DT>(row, V, aligned, rs, out);
    }
    return;
  }

  // ------------------------------------------------------------- publish
  RowPub* const pub = a.pubs + cta;
  if (tid == 0) {
    const bool xok = xtok >= 0 && xtok < V;
    const float xp = (!bad && paired && xok) ? prob_of<DT>(rs, sh.xbits[0], xtok) : 0.f;
    pub->rs = rs;
    pub->xprob = xp;
    if (role == ROLE_P && a.out_p) a.out_p[static_cast<size_t>(b) * kq + pos] = xp;
    if (role == ROLE_Q && a.out_q) a.out_q[static_cast<size_t>(b) * kq + pos] = xp;
    const uint32_t st = (bad ? SPEC_STATUS_BAD_ROW : 0u) | ((role == ROLE_P && !xok) ? SPEC_STATUS_BAD_TOKEN : 0u);
    if (st) set_status(a.status, st);
  }
  if (role == ROLE_P || role == ROLE_BONUS) {  // the vectors holding kept tokens, in index order
    uint32_t mine = 0u, nk = 0u;
    if (fast) {
      for (int i0 = 0; i0 < ngat; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t t = i < ngat ? wg[i] : 0u;
        const bool keep = i < ngat && tag_key(t) >= rs.kstar;
        const unsigned ball = __ballot_sync(kFull, keep);
        if (keep) wg[nk + __popc(ball & ((1u << lane) - 1u))] = t;
        nk += __popc(ball);
        __syncwarp();
      }
      mine = nk;
    }
    if (lane == 0) sh.w_u[warp][0] = mine;
    __syncthreads();
    uint32_t off = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) off += sh.w_u[w][0];
      tot += sh.w_u[w][0];
    }
    const bool listed = fast && !rs.all_kept && !bad && tot <= static_cast<uint32_t>(kPubList);
    if (listed)
      for (uint32_t i = lane; i < mine; i += 32) pub->list[off + i] = static_cast<uint32_t>(sg.beg) + tag_local(wg[i]);
    if (tid == 0) pub->nlist = listed ? tot : kPubReread;
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    sh.second = atomicAdd(a.seq_tickets + b, 1u) == static_cast<uint32_t>(2 * kq) ? 1 : 0;
  }
  __syncthreads();
  if (!sh.second) return;

  // ------------- the last row of sequence b: the first-rejection rule
  // (every position tested by its own thread, so the reads overlap)
  __threadfence();
  {
    const int k = kq;
    const int32_t* x = a.tokens + static_cast<size_t>(b) * k;
    int rej = k;  // this thread's position if it is rejected
    if (tid < k) {
      const RowPub* pp = a.pubs + 2 * (static_cast<size_t>(b) * k + tid);
      const float px = __ldcg(&pp[0].xprob), qx = __ldcg(&pp[1].xprob);
      const int bp = __ldcg(&pp[0].rs.bad), bq = __ldcg(&pp[1].rs.bad);
      const float u = a.uniforms[static_cast<size_t>(b) * (k + 2) + tid];
      const bool xok = x[tid] >= 0 && x[tid] < V;
      const bool acc = !bp && !bq && xok && u * qx < px;
      if (!acc) rej = tid;
    }
    // k <= 31: the first warp holds every position
    if (warp == 0) {
      const unsigned rb = __ballot_sync(kFull, rej < k);
      if (lane == 0) sh.draw_chunk = rb ? __ffs(rb) - 1 : k;
    }
    __syncthreads();
    const int n = sh.draw_chunk;
    int32_t* out = a.out_tokens + static_cast<size_t>(b) * (k + 1);
    if (tid < n) out[tid] = x[tid];
    else if (tid > n && tid <= k) out[tid] = -1;  // out[n]: drawn below, or by the draw kernel
    if (tid == 0) {
      a.out_n[b] = n;
      a.seq_tickets[b] = 0u;  // left zeroed for the next call
    }
  }

  // ------- the draw at n, here when the target row's kept vectors are listed
  {
    const int k = kq, n = sh.draw_chunk;
    const bool want_q = n < k;
    const RowPub* const pp = want_q ? a.pubs + 2 * (static_cast<size_t>(b) * k + n) : a.pubs + 2 * static_cast<size_t>(a.B) * k + b;
    const RowStat rp = ldcg_rowstat(&pp[0].rs);
    const RowStat rq = want_q ? ldcg_rowstat(&pp[1].rs) : rp;
    const uint32_t nlist = __ldcg(&pp[0].nlist);
    const bool listed = !rp.bad && !(want_q && rq.bad) && nlist != kPubReread && !rp.all_kept;
    if (!listed) return;  // the draw kernel draws over the whole rows
    const size_t rb = static_cast<size_t>(V) * E::kBytes;
    const unsigned char* const rowp =
        static_cast<const unsigned char*>(a.target) + (static_cast<size_t>(b) * (k + 1) + n) * rb;
    const unsigned char* const rowq =
        want_q ? static_cast<const unsigned char*>(a.draft) + (static_cast<size_t>(b) * k + n) * rb : rowp;
    const bool ap = a.aligned_target != 0, aq = want_q ? a.aligned_draft != 0 : ap;
    const float u = a.uniforms[static_cast<size_t>(b) * (k + 2) + (want_q ? k + 1 : k)];
    uint32_t* const idx = ltags;  // (the tags region is free now)
    float* const ew = reinterpret_cast<float*>(ltags + kPubList);
    uint32_t* const nls = ltags + 3 * kPubList;
    if (tid < 2 * k + 1)
      nls[tid] = __ldcg(&(tid < 2 * k ? a.pubs + 2 * static_cast<size_t>(b) * k + tid
                                        : a.pubs + 2 * static_cast<size_t>(a.B) * k + b)->nlist);
    const int token = draw_listed<DT>(sh, rp, rq, rowp, rowq, ap, aq, V, want_q, pp[0].list, static_cast<int>(nlist), u,
                                      idx, ew);
    if (tid == 0) {
      a.out_tokens[static_cast<size_t>(b) * (k + 1) + n] = token;
      a.draw_tickets[b] = kDrawnInTail;
    }
    clear_sequence_pubs(a, b, nls);
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 4) tail_kernel(const SampleArgs a) {
  __shared__ Shm sh;
  extern __shared__ __align__(16) uint32_t dsm[];
  tail_row<DT>(a, sh, dsm, static_cast<int>(blockIdx.x), false);
}

// ----------------------------------------------------- fused stream + tail
// One cooperative launch of as many CTAs as fit on the GPU at once, taking
// work items in order from a counter: the stream part of every row, then the
// tail part of every row.  A tail item waits for its row's stream item,
// which a running CTA took earlier and finishes without waiting on anyone;
// the tails of the first rows thus run beside the streams of the last ones,
// and no CTA slot idles between the two.  (Interleaving the two kinds
// earlier measured slower.)  The wait is bounded (about kMaxPolls polls):
// past it the row is published as bad and SPEC_STATUS_TIMEOUT is set.
constexpr int kMaxPolls = 1 << 22;

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 4) fused_kernel(const SampleArgs a) {
  __shared__ Shm sh;
  __shared__ int s_item, s_ok;
  extern __shared__ __align__(16) uint32_t dsm[];
  const int R = a.mode == MODE_SAMPLE ? a.B * (2 * a.k + 1) : a.B;
  const int tid = threadIdx.x;
  for (;;) {
    __syncthreads();  // the previous item is done with shared memory
    if (tid == 0) s_item = static_cast<int>(atomicAdd(a.work, 1u));
    __syncthreads();
    const int item = s_item;
    if (item >= 2 * R) break;
    // item -> (stream or tail, row)
    const int kind = item < R ? 0 : 1;
    const int rowi = item < R ? item : item - R;
    if (kind == 0) {
      const int item_row = rowi;
      stream_row<DT>(a, sh, dsm, item_row);
      __syncthreads();
      if (tid == 0 && a.launch_mode != SPEC_LAUNCH_FUSED_WAIT_TEST) {
        __threadfence();
        st_release_u32(a.done + item_row, 1u);
      }
    } else {
      const int r = rowi;
      if (tid == 0) {
        int ok = 0;
        for (int i = 0; i < a.poll_limit; ++i) {
          if (ld_acquire_u32(a.done + r)) {
            ok = 1;
            break;
          }
          __nanosleep(64);
        }
        if (!ok) set_status(a.status, SPEC_STATUS_TIMEOUT);
        a.done[r] = 0u;  // left zeroed for the next call
        s_ok = ok;
      }
      __syncthreads();
      tail_row<DT>(a, sh, dsm, r, s_ok == 0);
    }
  }
  // the last CTA out leaves the counters zeroed for the next call
  if (tid == 0 && atomicAdd(a.work + 1, 1u) == gridDim.x - 1) {
    a.work[0] = 0u;
    a.work[1] = 0u;
  }
}

// ------------------------------------------------------------ draw kernel
// After the tail kernel: sequence b's token at its first rejection n when the
// tail kernel could not draw it from listed vectors (no filter, a row the
// candidates did not decide, a non-finite row): drawn from max(0, p_n - q_n)
// with u_{k+1} (n < k) or from p_k with u_k (n = k), falling back to p_n
// when the residual has no mass.  a.chunks CTAs each sum one chunk of the
// whole rows; the last of them picks the chunk holding u * S from the chunk
// sums in order and walks it.
template <int DT>
__global__ void __launch_bounds__(kThreads, 4) draw_kernel(const SampleArgs a) {
  using E = Elt<DT>;
  __shared__ Shm sh;
  const int S = a.chunks;
  const int b = static_cast<int>(blockIdx.x) / S, s = static_cast<int>(blockIdx.x) % S;
  const int k = a.k, V = a.V, tid = threadIdx.x;
  if (__ldcg(a.draw_tickets + b) & kDrawnInTail) {  // drawn in the tail kernel: the last CTA resets the flag
    if (tid == 0) {
      const uint32_t old = atomicAdd(a.draw_tickets + b, 1u);
      if ((old & ~kDrawnInTail) == static_cast<uint32_t>(S - 1)) a.draw_tickets[b] = 0u;
    }
    return;
  }
  const int nvec = (V + E::kPerVec - 1) / E::kPerVec;
  const int n = min(max(a.out_n[b], 0), k);  // (written by the tail kernel; kept in range regardless)
  const bool want_q = n < k;
  const RowPub* const pp = want_q ? a.pubs + 2 * (static_cast<size_t>(b) * k + n) : a.pubs + 2 * static_cast<size_t>(a.B) * k + b;
  const RowStat rp = pp[0].rs;
  const RowStat rq = want_q ? pp[1].rs : rp;
  const size_t rb = static_cast<size_t>(V) * E::kBytes;
  const unsigned char* const rowp = static_cast<const unsigned char*>(a.target) + (static_cast<size_t>(b) * (k + 1) + n) * rb;
  const unsigned char* const rowq =
      want_q ? static_cast<const unsigned char*>(a.draft) + (static_cast<size_t>(b) * k + n) * rb : rowp;
  const bool ap = a.aligned_target != 0, aq = want_q ? a.aligned_draft != 0 : ap;
  const bool bad = rp.bad || (want_q && rq.bad);
  const float u = a.uniforms[static_cast<size_t>(b) * (k + 2) + (want_q ? k + 1 : k)];
  const int N = bad ? 0 : nvec;
  auto chunk_beg = [&](int cc) { return static_cast<int>(static_cast<long long>(N) * cc / S); };

  range_sums<DT>(sh, rp, rq, rowp, rowq, ap, aq, V, want_q, nullptr, chunk_beg(s), chunk_beg(s + 1));
  if (tid == 0) {
    DF sr{0.f, 0.f}, spp{0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      sr = df_add(sr, sh.w_s[w]);
      spp = df_add(spp, sh.w_sp[w]);
    }
    float* cs = a.csums + (static_cast<size_t>(b) * kMaxDrawChunks + s) * kChunkRec;
    cs[0] = sr.hi;
    cs[1] = sr.lo;
    cs[2] = spp.hi;
    cs[3] = spp.lo;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {  // kept for the walk of the chosen chunk
      cs[4 + w] = sh.w_s[w];
      cs[4 + kWarps + w] = sh.w_sp[w];
    }
    __threadfence();
    sh.second = atomicAdd(a.draw_tickets + b, 1u) == static_cast<uint32_t>(S - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!sh.second) return;

  // ------------------------ the last chunk of sequence b: pick one, walk it
  __shared__ float s_cs[kMaxDrawChunks * 4];
  __threadfence();
  if (tid < 4 * S) s_cs[tid] = __ldcg(a.csums + (static_cast<size_t>(b) * kMaxDrawChunks + tid / 4) * kChunkRec + tid % 4);
  __syncthreads();
  if (tid == 0) {
    const float* cs = s_cs;
    DF tr{0.f, 0.f}, tp{0.f, 0.f};
    for (int cc = 0; cc < S; ++cc) {
      tr = df_add2(tr, DF{cs[4 * cc], cs[4 * cc + 1]});
      tp = df_add2(tp, DF{cs[4 * cc + 2], cs[4 * cc + 3]});
    }
    const bool use_q = want_q && tr.hi > 0.f;  // a residual with no mass: draw from p
    const DF target = df_mul_f(use_q ? tr : tp, u);
    DF run{0.f, 0.f}, base{0.f, 0.f}, lbase{0.f, 0.f};
    int csel = -1, clast = -1;
    const int o = use_q ? 0 : 2;
    for (int cc = 0; cc < S; ++cc) {
      const DF sc{cs[4 * cc + o], cs[4 * cc + o + 1]};
      const DF nxt = df_add2(run, sc);
      if (sc.hi > 0.f) { clast = cc; lbase = run; }
      if (csel < 0 && sc.hi > 0.f && df_lt(target, nxt)) { csel = cc; base = run; }
      run = nxt;
    }
    if (csel < 0) { csel = clast; base = lbase; }
    sh.draw_chunk = bad ? -1 : csel;
    sh.draw_useq = use_q ? 1 : 0;
    sh.draw_target = df_add2(target, df_neg(base));
  }
  __syncthreads();
  const int cs = sh.draw_chunk;
  int token = -1;
  if (cs >= 0) {
    const bool use_q = sh.draw_useq != 0;
    // the chosen chunk's per-warp sums, as its CTA recorded them
    if (cs != s && tid < 2 * kWarps) {
      const float v = __ldcg(a.csums + (static_cast<size_t>(b) * kMaxDrawChunks + cs) * kChunkRec + 4 + tid);
      if (tid < kWarps) sh.w_s[tid] = v;
      else sh.w_sp[tid - kWarps] = v;
    }
    __syncthreads();
    token = range_walk<DT>(sh, rp, rq, rowp, rowq, ap, aq, V, use_q, sh.draw_target, nullptr, chunk_beg(cs),
                           chunk_beg(cs + 1));
  }
  if (tid == 0) a.out_tokens[static_cast<size_t>(b) * (k + 1) + n] = token;
  // leave the workspace zeroed for the next call, whatever its shape
  for (int i = tid; i < kChunkRec * S; i += kThreads) a.csums[static_cast<size_t>(b) * kMaxDrawChunks * kChunkRec + i] = 0.f;
  if (tid == 0) a.draw_tickets[b] = 0u;
  clear_sequence_pubs(a, b, nullptr);
}

// ------------------------------------------------------------------ launch

size_t stream_smem_bytes(bool filter) { return filter ? kWarps * kLaneTags * 32 * sizeof(uint32_t) : 16; }
size_t sample_smem_bytes(int dtype, bool filter) {
  (void)dtype;
  return filter ? (kRowTags + kWindow + kWarps * kBmapWords) * sizeof(uint32_t) : 16;
}

template <int DT>
static int launch_all(const SampleArgs& args, cudaStream_t st) {
  SampleArgs a = args;
  a.poll_limit = a.launch_mode == SPEC_LAUNCH_FUSED_WAIT_TEST ? 64 : kMaxPolls;
  const bool filter = a.top_k > 0 || a.top_p < 1.f;
  const int rows = a.mode == MODE_SAMPLE ? a.B * (2 * a.k + 1) : a.B;
  const size_t s1 = stream_smem_bytes(filter), s2 = sample_smem_bytes(DT, filter);
  static_assert(kRowTags * 4 + (kWindow + kWarps * kBmapWords) * 4 <= 48 * 1024, "tail kernel shared memory");
  // stream and tail fused in one cooperative launch when the GPU allows it
  bool fused = false;
  if (a.launch_mode != SPEC_LAUNCH_SEPARATE) {
    const size_t sf = s1 > s2 ? s1 : s2;
    int per_sm = 0, dev = 0, coop = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_kernel<DT>, kThreads, sf) == cudaSuccess &&
        per_sm > 0) {
      const int grid = std::min(per_sm * num_sms(), 2 * rows);
      void* params[] = {&a};
      fused = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fused_kernel<DT>), dim3(grid), dim3(kThreads),
                                          params, sf, st) == cudaSuccess;
    }
    if (!fused) (void)cudaGetLastError();  // (clear a refused launch; the two launches below stand in)
  }
  if (!fused) {
    stream_kernel<DT><<<rows, kThreads, s1, st>>>(a);
    tail_kernel<DT><<<rows, kThreads, s2, st>>>(a);
  }
  if (a.mode == MODE_SAMPLE) draw_kernel<DT><<<a.B * a.chunks, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

int launch_sample(const SampleArgs& a, int dtype, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == DT_BF16) return launch_all<DT_BF16>(a, st);
  if (dtype == DT_F32) return launch_all<DT_F32>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace specv
