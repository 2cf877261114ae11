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
// How (one GPU, memory-bound).  One persistent cooperative launch takes work
// items from a counter: every row of every sequence (sequence by sequence),
// then the chunks of the draws that need whole rows.  A row's CTA reads the
// row from HBM once, 16-byte non-allocating loads, four in flight per thread:
//   - masses sit on a power-of-two lattice: with c = log2(e) / T and an
//     integer K >= max(l) * c (raised, with an exact power-of-two rescale,
//     whenever the row maximum seen so far rises), mass(l) = 2^(l c - K),
//     one packed f32x2 fma and one ex2 per element; 2^(l c - K) / Z is the
//     softmax of l / T.
//   - a vector whose maximum reaches the window bottom (kDelta octaves of
//     mass below the row maximum seen so far) is queued in its warp; full
//     queues are counted element by element, 32 vectors at a time, into a
//     histogram of exact values (a ring over the value key), and their
//     first kListCap vectors are kept with their index.
// The tail scans the histogram from the top for the top-k and top-p cut (a
// token is kept while the mass ranked before it is below top_p times the
// top-k mass), the number of tokens of the cut value that are kept (lowest
// indices first) and the kept normaliser.  The kept vectors give the index
// bound of that tie and, for target rows, the row vectors holding kept
// tokens in index order.  A row whose cut lies below the window (or an fp32
// row, whose values are not counted exactly) takes an exact search that
// re-reads it.  The last row of a sequence to finish (ticket, no wait) tests
// u_i q_i(x_i) < p_i(x_i) at every position, takes the first rejection n,
// commits the accepted prefix and draws the token at n over the target row's
// listed kept vectors; rows without such a list (no filter, dense kept sets)
// are queued for a draw over whole rows in chunks.
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

constexpr float kDelta = 16.f;      // octaves of mass below the row maximum the histogram window spans
constexpr int kTieCap = 1024;       // tokens of the cut value gathered to find the tie's index bound
constexpr int kTieRankMax = 256;    // above this many, the bound is found by a pass over the row
constexpr int kMaxPolls = 1 << 22;  // polls before a wait of the fused kernel gives up

// Dynamic shared memory of a row CTA (filtered bf16 rows): the histogram
// ring, the per-warp candidate queues (data, index) and the kept candidate
// list (data, index).  After the stream the histogram holds the tie tokens
// and the draw scratch, and the queues the kept-vector bitmap.
constexpr size_t kHistBytes = sizeof(uint32_t) * kRing;
constexpr size_t kQDataOff = kHistBytes;
constexpr size_t kQIdxOff = kQDataOff + sizeof(uint4) * kWarps * kQCap;
constexpr size_t kListOff = kQIdxOff + sizeof(uint32_t) * kWarps * kQCap;
constexpr size_t kListIdxOff = kListOff + sizeof(uint4) * kListCap;
constexpr size_t kRowSmem = kListIdxOff + sizeof(uint32_t) * kListCap;
constexpr size_t kBitmapBytes = kListOff - kQDataOff;  // kept-vector bitmap in the queues' place
static_assert(kHistBytes >= sizeof(uint32_t) * 3 * kPubList, "draw scratch in the histogram's place");
static_assert(kHistBytes >= sizeof(uint32_t) * kTieCap, "tie tokens in the histogram's place");

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

// Shared state of one CTA (static shared memory).
struct Shm {
  float w_s[kWarps];           // per-warp sums (reductions, draw weights)
  float w_sp[kWarps];
  uint32_t w_u[kWarps][2];
  uint32_t wm[2][kWarps];      // per-warp running maxima at window updates (double-buffered)
  DF wz[kWarps];               // per-warp row sums
  uint32_t sc_cnt[kWarps];     // key scan: per-warp counts and masses
  double sc_mass[kWarps];
  int nlist;                   // candidate vectors appended to the list (may exceed kListCap)
  int ntie;                    // tokens of the cut value gathered
  int nkept;                   // kept vectors of a target row
  // row results passed between the threads of the CTA
  uint32_t mbits;              // bits of the row maximum
  float K;                     // lattice exponent at the end of the stream
  DF z;                        // row sum
  int corrupt;                 // the histogram window is not valid
  uint32_t kb;                 // lowest key counted by the histogram
  uint32_t vk;                 // top-k cut: key, kept tokens of that value, tokens of that value
  int ck, cnt_vk;
  double zk;                   // mass of the top-k set
  uint32_t vstar;              // top-p cut: key, kept, total, kept mass
  int jstar, cnt_vstar;
  double zkept;
  int found;
  int tie_idx;
  uint32_t xbits;              // the row's value at the draft token
  int second;                  // the last row of its sequence / the last chunk of its draw
  int item;
  int flag;
  // the draw
  int draw_warp;
  float draw_base;
  int draw_token;
  int draw_useq;
  int draw_chunk;
  DF draw_target;
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


// ------------------------------------------------------------ work items
constexpr int ROLE_P = 0;      // target row of a draft position
constexpr int ROLE_Q = 1;      // draft row of a draft position
constexpr int ROLE_BONUS = 2;  // target row after the last draft
constexpr int ROLE_PROBS = 3;  // one row of spec_transform_probs

// Row item `item`: sequence by sequence, the target and draft rows of each
// draft position, then the bonus target row (MODE_PROBS: row `item`).
// `pub` is the row's record: 2 (b k + i) + role for draft positions, 2 B k + b
// for the bonus rows.
struct RowRef {
  int role, b, pos, pub;
  const unsigned char* row;
  bool aligned;
};
template <int DT>
__device__ __forceinline__ RowRef row_ref(const SampleArgs& a, int item) {
  using E = Elt<DT>;
  const unsigned char* tgt = static_cast<const unsigned char*>(a.target);
  const size_t rb = static_cast<size_t>(a.V) * E::kBytes;
  RowRef r;
  if (a.mode == MODE_PROBS) {
    r.role = ROLE_PROBS;
    r.b = item;
    r.pos = 0;
    r.pub = item;
    r.row = tgt + static_cast<size_t>(item) * rb;
    r.aligned = a.aligned_target != 0;
    return r;
  }
  const int k = a.k;
  r.b = item / (2 * k + 1);
  const int j = item - r.b * (2 * k + 1);
  if (j < 2 * k) {
    r.role = (j & 1) ? ROLE_Q : ROLE_P;
    r.pos = j >> 1;
    r.pub = 2 * (r.b * k + r.pos) + (j & 1);
    r.row = r.role == ROLE_P ? tgt + (static_cast<size_t>(r.b) * (k + 1) + r.pos) * rb
                             : static_cast<const unsigned char*>(a.draft) + (static_cast<size_t>(r.b) * k + r.pos) * rb;
    r.aligned = (r.role == ROLE_P ? a.aligned_target : a.aligned_draft) != 0;
  } else {
    r.role = ROLE_BONUS;
    r.pos = k;
    r.pub = 2 * a.B * k + r.b;
    r.row = tgt + (static_cast<size_t>(r.b) * (k + 1) + k) * rb;
    r.aligned = a.aligned_target != 0;
  }
  return r;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_shared_u32(uint32_t a) {
  asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(a) : "memory");
}
__device__ __forceinline__ uint32_t hmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Running maximum of a thread, as bits: bf16x2 (both halves), or f32.
template <int DT>
struct RunMax;
template <>
struct RunMax<DT_BF16> {
  static constexpr uint32_t kNeg = 0xFF80FF80u;
  __device__ static __forceinline__ uint32_t vec(const uint4& x) {
    const uint32_t m = hmax2(hmax2(x.x, x.y), hmax2(x.z, x.w));
    return hmax2(m, __byte_perm(m, 0, 0x1032));
  }
  __device__ static __forceinline__ uint32_t join(uint32_t a, uint32_t b) { return hmax2(a, b); }
  __device__ static __forceinline__ uint32_t bits(uint32_t m) { return m & 0xFFFFu; }
  __device__ static __forceinline__ float value(uint32_t m) { return __uint_as_float(m & 0xFFFF0000u); }
};
template <>
struct RunMax<DT_F32> {
  static constexpr uint32_t kNeg = 0xFF800000u;
  __device__ static __forceinline__ uint32_t vec(const uint4& x) {
    return __float_as_uint(max_nan(max_nan(__uint_as_float(x.x), __uint_as_float(x.y)),
                                   max_nan(__uint_as_float(x.z), __uint_as_float(x.w))));
  }
  __device__ static __forceinline__ uint32_t join(uint32_t a, uint32_t b) {
    return __float_as_uint(max_nan(__uint_as_float(a), __uint_as_float(b)));
  }
  __device__ static __forceinline__ uint32_t bits(uint32_t m) { return m; }
  __device__ static __forceinline__ float value(uint32_t m) { return __uint_as_float(m); }
};

// ---------------------------------------------------------------- stream
// One row streamed once by the CTA (see the file comment).  Leaves in sh:
// mbits (row maximum), K, z (row sum of 2^(l c - K)), and for FILT the
// histogram window (kb, corrupt), the candidate list (nlist) and their data
// in dsm.
template <int DT, bool FILT>
__device__ __noinline__ void stream_row(const unsigned char* row, int V, bool aligned, float c, Shm& sh,
                                        unsigned char* dsm) {
  using E = Elt<DT>;
  using M = RunMax<DT>;
  constexpr int U = kStreamU;
  constexpr int PV = E::kPerVec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = (V + PV - 1) / PV;
  constexpr int kStep = kThreads * U;
  const int iters = (nvec + kStep - 1) / kStep;
  const uint32_t hbase = smem_addr(dsm);
  const uint32_t qd = smem_addr(dsm + kQDataOff) + warp * kQCap * 16;
  const uint32_t qi = smem_addr(dsm + kQIdxOff) + warp * kQCap * 4;
  uint4* const ldata = reinterpret_cast<uint4*>(dsm + kListOff);
  uint32_t* const lidx = reinterpret_cast<uint32_t*>(dsm + kListIdxOff);
  const uint4 pad = make_uint4(Hot<DT>::kPad, Hot<DT>::kPad, Hot<DT>::kPad, Hot<DT>::kPad);
  if (FILT) {
    uint32_t* hist = reinterpret_cast<uint32_t*>(dsm);
    for (int i = tid; i < kRing; i += kThreads) hist[i] = 0u;
    if (tid == 0) {
      sh.nlist = 0;
      sh.corrupt = 0;
    }
  }
  uint4 cur[U], nxt[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int v = u * kThreads + tid;
    cur[u] = v < nvec ? load_vec<DT>(row, v, V, aligned) : pad;
  }
  uint32_t mx = M::kNeg;
#pragma unroll
  for (int u = 0; u < U; ++u) mx = M::join(mx, M::vec(cur[u]));

  // window and lattice state (the same in every thread)
  float K = 0.f, lbf = __int_as_float(0x7F800000);  // +inf: nothing is a candidate until anchored
  bool anchored = false, lbpos = false;
  uint32_t ktop = 0u, kb = 0u;
  int corrupt = 0;
  u64 nk2 = pkf(-0.f, -0.f);
  const u64 c2 = pkf(c, c);
  u64 acc0 = pkf(0.f, 0.f), acc1 = pkf(0.f, 0.f);
  int par = 0;
  uint32_t qn = 0u, qf = 0u;
  const uint32_t ltmask = (1u << lane) - 1u;

  // The window update: every thread takes the CTA maximum seen so far; a
  // higher maximum raises K (exact rescale of the partial sums), the window
  // bottom (its departing slots cleared) and the anchor.
  auto update = [&]() {
    uint32_t m1 = mx;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m1 = M::join(m1, __shfl_xor_sync(kFull, m1, o));
    if (lane == 0) sh.wm[par][warp] = m1;
    __syncthreads();
    uint32_t m = sh.wm[par][0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) m = M::join(m, sh.wm[par][w]);
    par ^= 1;
    const uint32_t mb = M::bits(m);
    const float mv = M::value(m);
    if (!isfinite(mv) || !(fabsf(mv * c) < 1073741824.f)) return;  // (bad rows are found at the end)
    const uint32_t nt = E::key(mb);
    if (anchored && nt <= ktop) return;
    const float nK = ceilf(mv * c);
    if (anchored) {
      const float s = exp2i(static_cast<int>(K - nK));
      const u64 s2 = pkf(s, s);
      acc0 = mul2(acc0, s2);
      acc1 = mul2(acc1, s2);
      if (FILT && nt > ktop + static_cast<uint32_t>(kFreeKeys)) corrupt = 1;
    }
    K = nK;
    nk2 = pkf(-K, -K);
    if (FILT && DT == DT_BF16) {
      uint32_t nkb = E::key(bits_round_up<DT>(mv - kDelta / c));
      if (nt >= static_cast<uint32_t>(kWinKeys - 1)) nkb = max(nkb, nt - static_cast<uint32_t>(kWinKeys - 1));
      if (anchored && nkb > kb) {  // departing keys: their slots are cleared (their masses stay in the sums)
        uint32_t* hist = reinterpret_cast<uint32_t*>(dsm);
        const uint32_t end = min(nkb, kb + static_cast<uint32_t>(kRing));
        for (uint32_t kk = kb + tid; kk < end; kk += kThreads) hist[kk & (kRing - 1)] = 0u;
      }
      if (!anchored || nkb > kb) {
        kb = nkb;
        lbf = value_of_key<DT>(kb);
        lbpos = lbf > 0.f;
      }
    }
    ktop = nt;
    anchored = true;
  };

  // Count queued vectors [e, e + 32) of this warp (lanes at or past `cnt`
  // idle) into the histogram and append them to the candidate list.
  auto flush = [&](uint32_t e0, uint32_t cnt) {
    __syncwarp();
    const bool has = static_cast<uint32_t>(lane) < cnt;
    uint4 d = make_uint4(0u, 0u, 0u, 0u);
    uint32_t vi = 0u;
    if (has) {
      const uint32_t slot = (e0 + lane) & (kQCap - 1);
      d = lds128(qd + slot * 16);
      vi = lds_u32(qi + slot * 4);
      const uint32_t w4[4] = {d.x, d.y, d.z, d.w};
      if (lbpos) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w = w4[j];
          if (__uint_as_float(w << 16) >= lbf) red_shared_u32(hbase + ((w << 2) & ((kRing - 1) << 2)));
          if (__uint_as_float(w & 0xFFFF0000u) >= lbf) red_shared_u32(hbase + ((w >> 14) & ((kRing - 1) << 2)));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t bj = (j & 1) ? (w4[j >> 1] >> 16) : (w4[j >> 1] & 0xFFFFu);
          if (E::value(bj) >= lbf) red_shared_u32(hbase + ((E::key(bj) & (kRing - 1)) << 2));
        }
      }
    }
    __syncwarp();
    int base = 0;
    if (lane == 0) base = atomicAdd(&sh.nlist, static_cast<int>(cnt));
    base = __shfl_sync(kFull, base, 0);
    if (has && base + lane < kListCap) {
      ldata[base + lane] = d;
      lidx[base + lane] = vi;
    }
  };

  if (FILT && DT == DT_BF16) update();
  else {
    // (unfiltered rows only need the lattice exponent: one update)
    update();
  }

  for (int it = 0; it < iters; ++it) {
    if (it + 1 < iters) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = (it + 1) * kStep + u * kThreads + tid;
        nxt[u] = v < nvec ? load_vec<DT>(row, v, V, aligned) : pad;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint4 x = cur[u];
      const uint32_t vm = M::vec(x);
      mx = M::join(mx, vm);
      Hot<DT>::mass_vec(x, c2, nk2, acc0, acc1);
      if (FILT && DT == DT_BF16) {
        const bool cand = M::value(vm) >= lbf;
        const uint32_t bal = __ballot_sync(kFull, cand);
        if (bal) {
          const uint32_t pos = qn + __popc(bal & ltmask);
          if (cand) {
            const uint32_t slot = pos & (kQCap - 1);
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(qd + slot * 16), "r"(x.x), "r"(x.y), "r"(x.z),
                         "r"(x.w)
                         : "memory");
            sts_u32(qi + slot * 4, static_cast<uint32_t>(it * kStep + u * kThreads + tid));
          }
          qn += __popc(bal);
          if (qn - qf >= 32u) {
            flush(qf, 32u);
            qf += 32u;
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) cur[u] = nxt[u];
    if (((it + 1) % kSyncEvery) == 0 && it + 1 < iters) update();
  }
  if (FILT && DT == DT_BF16 && qn != qf) flush(qf, qn - qf);

  // the row maximum and sum
  {
    uint32_t m1 = mx;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m1 = M::join(m1, __shfl_xor_sync(kFull, m1, o));
    float a0, a1, a2, a3;
    upk(acc0, a0, a1);
    upk(acc1, a2, a3);
    DF z{(a0 + a1) + (a2 + a3), 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z = df_add2(z, DF{__shfl_xor_sync(kFull, z.hi, o), __shfl_xor_sync(kFull, z.lo, o)});
    if (lane == 0) {
      sh.wm[par][warp] = m1;
      sh.wz[warp] = z;
    }
    if (FILT && tid == 0) {
      sh.kb = kb;
      if (!anchored) corrupt = 1;
      sh.corrupt = corrupt;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t m = sh.wm[par][0];
      DF t{0.f, 0.f};
      for (int w = 0; w < kWarps; ++w) {
        m = M::join(m, sh.wm[par][w]);
        t = df_add2(t, sh.wz[w]);
      }
      const float mv = M::value(m);
      float Kf = K;
      if (isfinite(mv) && fabsf(mv * c) < 1073741824.f) {
        Kf = ceilf(mv * c);
        if (Kf > K) {  // elements above the last anchor: exact rescale to the final exponent
          const float s = exp2i(static_cast<int>(K - Kf));
          t = DF{t.hi * s, t.lo * s};
        }
        if (FILT && (!anchored || E::key(M::bits(m)) > ktop + static_cast<uint32_t>(kFreeKeys))) sh.corrupt = 1;
      }
      sh.mbits = M::bits(m);
      sh.K = Kf;
      sh.z = t;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------- the cut from the ring
// Exclusive CTA scan (thread order) of a count and a mass; totals too.
__device__ __forceinline__ void block_scan_cm(Shm& sh, uint32_t c, double m, uint32_t& cb, double& mb, uint32_t& ct,
                                              double& mt) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t ci = c;
  double mi = m;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t co = __shfl_up_sync(kFull, ci, o);
    const double mo = __shfl_up_sync(kFull, mi, o);
    if (lane >= o) {
      ci += co;
      mi += mo;
    }
  }
  if (lane == 31) {
    sh.sc_cnt[warp] = ci;
    sh.sc_mass[warp] = mi;
  }
  __syncthreads();
  uint32_t wc = 0u, tc = 0u;
  double wmass = 0.0, tm = 0.0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) {
      wc += sh.sc_cnt[w];
      wmass += sh.sc_mass[w];
    }
    tc += sh.sc_cnt[w];
    tm += sh.sc_mass[w];
  }
  __syncthreads();
  cb = wc + ci - c;
  mb = wmass + (mi - m);
  ct = tc;
  mt = tm;
}

// The top-k / top-p cut from the histogram ring (keys kb .. kmax).  Fills
// rs.kstar, rs.keep, rs.total and *zkept.  False when the cut may lie below
// the window (the caller then searches the whole row).  Whole CTA.
template <int DT>
__device__ __noinline__ bool cut_from_hist(Shm& sh, const uint32_t* hist, RowStat& rs, int top_k, float top_p,
                                           double zfull, uint32_t kb, double* zkept) {
  const int tid = threadIdx.x;
  const bool topk_on = top_k > 0, topp_on = top_p < 1.f;
  const uint32_t kmax = rs.kmax;
  if (kmax < kb) return false;
  const int nk = static_cast<int>(kmax - kb) + 1;
  if (nk > kRing) return false;
  const int per = (nk + kThreads - 1) / kThreads;
  const int i0 = min(nk, tid * per), i1 = min(nk, i0 + per);
  uint32_t cnt = 0u;
  double mass = 0.0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = kmax - static_cast<uint32_t>(i);
    const uint32_t n = hist[key & (kRing - 1)];
    if (n) {
      cnt += n;
      mass += static_cast<double>(n) * static_cast<double>(lat_mass(value_of_key<DT>(key), rs.c, rs.K));
    }
  }
  if (tid == 0) sh.found = 0;
  uint32_t cb, ct;
  double mb, mt;
  block_scan_cm(sh, cnt, mass, cb, mb, ct, mt);
  // top-k: the value holding the top_k-th token
  double zk = zfull;
  uint32_t vk = 0u;
  int ck = 0;
  if (topk_on) {
    if (ct < static_cast<uint32_t>(top_k)) return false;  // (uniform: every thread has the totals)
    if (cb < static_cast<uint32_t>(top_k) && cb + cnt >= static_cast<uint32_t>(top_k)) {
      uint32_t rc = cb;
      double rm = mb;
      for (int i = i0; i < i1; ++i) {
        const uint32_t key = kmax - static_cast<uint32_t>(i);
        const uint32_t n = hist[key & (kRing - 1)];
        if (!n) continue;
        const double w = static_cast<double>(lat_mass(value_of_key<DT>(key), rs.c, rs.K));
        if (rc + n >= static_cast<uint32_t>(top_k)) {
          sh.vk = key;
          sh.ck = top_k - static_cast<int>(rc);
          sh.cnt_vk = static_cast<int>(n);
          sh.zk = rm + static_cast<double>(top_k - static_cast<int>(rc)) * w;
          break;
        }
        rc += n;
        rm += static_cast<double>(n) * w;
      }
    }
    __syncthreads();
    zk = sh.zk;
    vk = sh.vk;
    ck = sh.ck;
  }
  if (!topp_on) {
    rs.kstar = vk;
    rs.keep = ck;
    rs.total = sh.cnt_vk;
    *zkept = zk;
    return true;
  }
  // top-p on the top-k set: the first value at which the mass ranked at or
  // above it reaches top_p * zk; its tokens are kept while the mass before
  // them is below that target
  const double target = static_cast<double>(top_p) * zk;
  if (!topk_on && mt < target) return false;
  if (mb < target && mb + mass >= target) {
    double rm = mb;
    for (int i = i0; i < i1; ++i) {
      const uint32_t key = kmax - static_cast<uint32_t>(i);
      const uint32_t n = hist[key & (kRing - 1)];
      if (!n) continue;
      const double w = static_cast<double>(lat_mass(value_of_key<DT>(key), rs.c, rs.K));
      if (rm + static_cast<double>(n) * w >= target || (topk_on && key <= vk)) {
        uint32_t vs = key, avail = n, tot = n;
        double before = rm;
        if (topk_on && key <= vk) {  // the crossing is at the top-k cut value, within its kept tokens
          const double wk = static_cast<double>(lat_mass(value_of_key<DT>(vk), rs.c, rs.K));
          vs = vk;
          avail = static_cast<uint32_t>(ck);
          tot = static_cast<uint32_t>(sh.cnt_vk);
          before = zk - static_cast<double>(ck) * wk;
        }
        const double ws = static_cast<double>(lat_mass(value_of_key<DT>(vs), rs.c, rs.K));
        double need = ws > 0.0 ? ceil((target - before) / ws) : static_cast<double>(avail);
        if (!(need >= 1.0)) need = 1.0;
        const uint32_t j = need >= static_cast<double>(avail) ? avail : static_cast<uint32_t>(need);
        sh.vstar = vs;
        sh.jstar = static_cast<int>(j);
        sh.cnt_vstar = static_cast<int>(tot);
        sh.zkept = before + static_cast<double>(j) * ws;
        sh.found = 1;
        break;
      }
      rm += static_cast<double>(n) * w;
    }
  }
  __syncthreads();
  if (!sh.found) return false;
  rs.kstar = sh.vstar;
  rs.keep = sh.jstar;
  rs.total = sh.cnt_vstar;
  *zkept = sh.zkept;
  return true;
}

// ------------------------------------------------ tokens of one value
// Tokens of key `kstar` among vectors [e0, e1) of a row with index < jmax.
// Whole CTA; every thread gets the count.
template <int DT>
__device__ __noinline__ uint32_t count_equal(Shm& sh, const unsigned char* row, int V, bool aligned, int e0, int e1,
                                             uint32_t kstar, int jmax) {
  using E = Elt<DT>;
  uint32_t cnt = 0u;
  constexpr int kU = 4;
  for (int v0 = e0 + static_cast<int>(threadIdx.x); v0 < e1; v0 += kU * kThreads) {
    uint4 xs[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = v0 + u * kThreads;
      xs[u] = v < e1 ? load_vec<DT>(row, v, V, aligned) : make_uint4(Hot<DT>::kPad, Hot<DT>::kPad, Hot<DT>::kPad, Hot<DT>::kPad);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = v0 + u * kThreads;
#pragma unroll
      for (int j = 0; j < E::kPerVec; ++j) {
        const int t = v * E::kPerVec + j;
        if (v < e1 && t < jmax && t < V && E::key(E::bits_of(xs[u], j)) == kstar) ++cnt;
      }
    }
  }
  return block_sum_u32(cnt, sh);
}

// Index of the m-th (1-based) token of key `kstar` among vectors [e0, e1) in
// index order, or -1.  Whole CTA: per-warp counts over equal parts, then the
// warp holding it walks its part 32 vectors at a time.
template <int DT>
__device__ __noinline__ int find_nth_equal(Shm& sh, const unsigned char* row, int V, bool aligned, int e0, int e1,
                                           uint32_t kstar, int m) {
  using E = Elt<DT>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Part pt = warp_part(e0, e1, warp);
  uint32_t cnt = 0u;
  for (int v = pt.beg + lane; v < pt.end; v += 32) {
    const uint4 x = load_vec<DT>(row, v, V, aligned);
#pragma unroll
    for (int j = 0; j < E::kPerVec; ++j)
      if (v * E::kPerVec + j < V && E::key(E::bits_of(x, j)) == kstar) ++cnt;
  }
  cnt = warp_sum_u32(cnt);
  if (lane == 0) sh.w_u[warp][0] = cnt;
  if (threadIdx.x == 0) sh.tie_idx = -1;
  __syncthreads();
  uint32_t before = 0u;
  for (int w = 0; w < warp; ++w) before += sh.w_u[w][0];
  if (before < static_cast<uint32_t>(m) && before + cnt >= static_cast<uint32_t>(m)) {
    uint32_t run = before;
    for (int v0 = pt.beg; v0 < pt.end; v0 += 32) {
      const int v = v0 + lane;
      uint4 x = make_uint4(Hot<DT>::kPad, Hot<DT>::kPad, Hot<DT>::kPad, Hot<DT>::kPad);
      if (v < pt.end) x = load_vec<DT>(row, v, V, aligned);
      uint32_t bits = 0u;
#pragma unroll
      for (int j = 0; j < E::kPerVec; ++j)
        if (v < pt.end && v * E::kPerVec + j < V && E::key(E::bits_of(x, j)) == kstar) bits |= 1u << j;
      const uint32_t lc = __popc(bits);
      const uint32_t incl = warp_incl_scan_u32(lc);
      const uint32_t tot = __shfl_sync(kFull, incl, 31);
      if (run + tot >= static_cast<uint32_t>(m)) {
        const uint32_t excl = incl - lc;
        if (run + excl < static_cast<uint32_t>(m) && run + incl >= static_cast<uint32_t>(m)) {
          uint32_t need = static_cast<uint32_t>(m) - run - excl;  // 1-based within this lane's vector
          int idx = -1;
#pragma unroll
          for (int j = 0; j < E::kPerVec; ++j)
            if (((bits >> j) & 1u) && idx < 0 && --need == 0u) idx = v * E::kPerVec + j;
          sh.tie_idx = idx;
        }
        break;
      }
      run += tot;
    }
  }
  __syncthreads();
  return sh.tie_idx;
}

// The index bound of a row's tie from its candidate list (every token of the
// cut value lies in a listed vector): the keep-th lowest index of the listed
// tokens of key kstar, plus one.  -1 when the list cannot tell.  Whole CTA.
template <int DT>
__device__ __noinline__ int tie_cut_from_list(Shm& sh, const unsigned char* dsm, uint32_t* tix, int nlist,
                                              uint32_t kstar, int keep, int total) {
  using E = Elt<DT>;
  const uint4* ldata = reinterpret_cast<const uint4*>(dsm + kListOff);
  const uint32_t* lidx = reinterpret_cast<const uint32_t*>(dsm + kListIdxOff);
  if (threadIdx.x == 0) {
    sh.ntie = 0;
    sh.tie_idx = -1;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < nlist; e += kThreads) {
    const uint4 d = ldata[e];
    const uint32_t v = lidx[e];
#pragma unroll
    for (int j = 0; j < E::kPerVec; ++j) {
      if (E::key(E::bits_of(d, j)) == kstar) {
        const int p = atomicAdd(&sh.ntie, 1);
        if (p < kTieCap) tix[p] = v * E::kPerVec + j;
      }
    }
  }
  __syncthreads();
  const int n = sh.ntie;
  if (n != total || n > kTieRankMax) return -1;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const uint32_t mine = tix[i];
    int r = 0;
    for (int j = 0; j < n; ++j) r += tix[j] < mine ? 1 : 0;
    if (r == keep - 1) sh.tie_idx = static_cast<int>(mine);
  }
  __syncthreads();
  return sh.tie_idx < 0 ? -1 : sh.tie_idx + 1;
}

// The vectors of a target row holding a token at or above value key kstar,
// in index order, from its candidate list (a bitmap over the row's vectors
// in the queues' place).  Returns their count (> kPubList: not listed).
template <int DT>
__device__ __noinline__ int kept_vectors(Shm& sh, unsigned char* dsm, int nlist, int nvec, uint32_t kstar,
                                         uint32_t* out) {
  using M = RunMax<DT>;
  const uint4* ldata = reinterpret_cast<const uint4*>(dsm + kListOff);
  const uint32_t* lidx = reinterpret_cast<const uint32_t*>(dsm + kListIdxOff);
  uint32_t* bm = reinterpret_cast<uint32_t*>(dsm + kQDataOff);
  const int nw = (nvec + 31) / 32;
  if (nw * 4 > static_cast<int>(kBitmapBytes)) return kPubList + 1;
  for (int i = threadIdx.x; i < nw; i += kThreads) bm[i] = 0u;
  __syncthreads();
  const float vs = value_of_key<DT>(kstar);
  for (int e = threadIdx.x; e < nlist; e += kThreads) {
    if (M::value(M::vec(ldata[e])) >= vs) {
      const uint32_t v = lidx[e];
      atomicOr(&bm[v >> 5], 1u << (v & 31u));
    }
  }
  __syncthreads();
  // ordered compaction: thread t takes words [t * per, (t + 1) * per)
  const int per = (nw + kThreads - 1) / kThreads;
  const int w0 = min(nw, static_cast<int>(threadIdx.x) * per), w1 = min(nw, w0 + per);
  uint32_t c = 0u;
  for (int i = w0; i < w1; ++i) c += __popc(bm[i]);
  uint32_t cb, ct;
  double mb, mt;
  block_scan_cm(sh, c, 0.0, cb, mb, ct, mt);
  if (ct <= static_cast<uint32_t>(kPubList)) {
    uint32_t o = cb;
    for (int i = w0; i < w1; ++i) {
      uint32_t bits = bm[i];
      while (bits) {
        const int l = __ffs(bits) - 1;
        bits &= bits - 1u;
        out[o++] = static_cast<uint32_t>(i * 32 + l);
      }
    }
  }
  return static_cast<int>(ct);
}

// ------------------------------------------------------------ one row
template <int DT>
__device__ __noinline__ void process_row(const SampleArgs& a, Shm& sh, unsigned char* dsm, const int item);

// The records sequence b's rows published (headers and kept-vector lists)
// and, with draw_recs, its whole-row draw records, zeroed once every reader
// is done: the workspace is left zero for the next call whatever its shape.
// Whole CTA.
__device__ __noinline__ void clear_sequence(const SampleArgs& a, int b, bool draw_recs) {
  const int k = a.k, nrows = 2 * k + 1, tid = threadIdx.x;
  auto pub_of = [&](int r) {
    return r < 2 * k ? a.pubs + 2 * static_cast<size_t>(b) * k + r : a.pubs + 2 * static_cast<size_t>(a.B) * k + b;
  };
  __syncthreads();
  for (int r = 0; r < nrows; ++r) {
    RowPub* p = pub_of(r);
    const uint32_t nl = __ldcg(&p->nlist);
    if (nl != kPubReread)
      for (uint32_t i = tid; i < nl && i < static_cast<uint32_t>(kPubList); i += kThreads) p->list[i] = 0u;
  }
  __syncthreads();
  constexpr int kHdrWords = static_cast<int>(offsetof(RowPub, list) / 4);
  for (int i = tid; i < nrows * kHdrWords; i += kThreads)
    reinterpret_cast<uint32_t*>(pub_of(i / kHdrWords))[i % kHdrWords] = 0u;
  if (draw_recs) {
    float* cs = a.csums + static_cast<size_t>(b) * kMaxDrawChunks * kChunkRec;
    for (int i = tid; i < kMaxDrawChunks * kChunkRec; i += kThreads) cs[i] = 0.f;
    for (int i = tid; i < 2 * kMaxDrawChunks; i += kThreads) {
      a.tcnt[static_cast<size_t>(b) * kMaxDrawChunks * 2 + i] = 0;
      a.tcut[static_cast<size_t>(b) * kMaxDrawChunks * 2 + i] = 0;
    }
  }
}

// The first-rejection rule and the draw for sequence b, run by the CTA that
// finished its last row.
template <int DT>
__device__ __noinline__ void finish_sequence(const SampleArgs& a, Shm& sh, unsigned char* dsm, const int b) {
  using E = Elt<DT>;
  const int k = a.k, V = a.V, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t* x = a.tokens + static_cast<size_t>(b) * k;
  __threadfence();
  int rej = k;
  if (tid < k) {
    const RowPub* pp = a.pubs + 2 * (static_cast<size_t>(b) * k + tid);
    const float px = __ldcg(&pp[0].xprob), qx = __ldcg(&pp[1].xprob);
    const int bp = __ldcg(&pp[0].rs.bad), bq = __ldcg(&pp[1].rs.bad);
    const float u = a.uniforms[static_cast<size_t>(b) * (k + 2) + tid];
    const bool xok = x[tid] >= 0 && x[tid] < V;
    if (!(!bp && !bq && xok && u * qx < px)) rej = tid;
  }
  if (warp == 0) {  // k <= 31: the first warp holds every position
    const unsigned rb = __ballot_sync(kFull, rej < k);
    if (lane == 0) sh.draw_chunk = rb ? __ffs(rb) - 1 : k;
  }
  __syncthreads();
  const int n = sh.draw_chunk;
  int32_t* out = a.out_tokens + static_cast<size_t>(b) * (k + 1);
  if (tid < n) out[tid] = x[tid];
  else if (tid <= k) out[tid] = -1;  // out[n]: written by the draw below or by the whole-row draw
  if (tid == 0) {
    a.out_n[b] = n;
    a.seq_tickets[b] = 0u;  // left zeroed for the next call
  }
  const bool want_q = n < k;
  const RowPub* const pp = want_q ? a.pubs + 2 * (static_cast<size_t>(b) * k + n) : a.pubs + 2 * static_cast<size_t>(a.B) * k + b;
  const RowStat rp = ldcg_rowstat(&pp[0].rs);
  const RowStat rq = want_q ? ldcg_rowstat(&pp[1].rs) : rp;
  const uint32_t nlist = __ldcg(&pp[0].nlist);
  const bool bad = rp.bad || (want_q && rq.bad);
  const bool q_known = !want_q || rq.all_kept || rq.tie_cut >= 0;
  const bool listed = !bad && !rp.all_kept && nlist != kPubReread && rp.tie_cut >= 0 && q_known;
  if (listed) {
    const size_t rb = static_cast<size_t>(V) * E::kBytes;
    const unsigned char* const rowp =
        static_cast<const unsigned char*>(a.target) + (static_cast<size_t>(b) * (k + 1) + n) * rb;
    const unsigned char* const rowq =
        want_q ? static_cast<const unsigned char*>(a.draft) + (static_cast<size_t>(b) * k + n) * rb : rowp;
    const bool ap = a.aligned_target != 0, aq = want_q ? a.aligned_draft != 0 : ap;
    const float u = a.uniforms[static_cast<size_t>(b) * (k + 2) + (want_q ? k + 1 : k)];
    uint32_t* const idx = reinterpret_cast<uint32_t*>(dsm);
    float* const ew = reinterpret_cast<float*>(dsm + sizeof(uint32_t) * kPubList);
    const int token = draw_listed<DT>(sh, rp, rq, rowp, rowq, ap, aq, V, want_q, pp[0].list, static_cast<int>(nlist), u,
                                      idx, ew);
    if (tid == 0) out[n] = token;
    clear_sequence(a, b, false);
  } else if (bad || a.launch_mode == SPEC_LAUNCH_FUSED_WAIT_TEST) {
    // nothing to draw (a non-finite row: token -1), or, in the wait test, a
    // draw whose queue entry is withheld so that its waits run out
    if (tid == 0 && !bad) atomicAdd(a.work + WK_QUEUED, 1u);
    clear_sequence(a, b, false);
  } else if (tid == 0) {
    // queued for the draw over whole rows (the queue counter first, so that a
    // claimer that sees every sequence finished sees the final count)
    const uint32_t e = atomicAdd(a.work + WK_QUEUED, 1u);
    st_release_u32(a.ready + e, static_cast<uint32_t>(b) + 1u);
  }
  if (tid == 0) {
    __threadfence();
    atomicAdd(a.work + WK_SEQS, 1u);
  }
}

template <int DT>
__device__ __noinline__ void process_row(const SampleArgs& a, Shm& sh, unsigned char* dsm, const int item) {
  using E = Elt<DT>;
  const RowRef rr = row_ref<DT>(a, item);
  const int role = rr.role, b = rr.b, pos = rr.pos;
  const unsigned char* const row = rr.row;
  const bool aligned = rr.aligned;
  const int tid = threadIdx.x;
  const int V = a.V;
  const float T = a.temperature_per_seq ? a.temperature_per_seq[b] : a.temperature;
  const bool bad_t = !(T > 0.f) || isinf(T) || isnan(T);
  const float c = bad_t ? 1.f : kLog2e / T;
  const int nvec = (V + E::kPerVec - 1) / E::kPerVec;
  const bool topk_on = a.top_k > 0, topp_on = a.top_p < 1.f;
  const bool filt = topk_on || topp_on;
  const bool paired = role == ROLE_P || role == ROLE_Q;
  const int xtok = paired ? a.tokens[static_cast<size_t>(b) * a.k + pos] : -1;
  const bool xok = xtok >= 0 && xtok < V;
  if (tid == 0) sh.xbits = xok ? E::bits_at(row, xtok) : 0u;  // (read early: its latency hides behind the stream)
  const bool hist_on = DT == DT_BF16 && filt && !bad_t;
  if (hist_on) stream_row<DT, true>(row, V, aligned, c, sh, dsm);
  else stream_row<DT, false>(row, V, aligned, c, sh, dsm);

  RowStat rs;
  rs.c = c;
  rs.K = sh.K;
  rs.m = E::value(sh.mbits);
  rs.kmax = E::key(sh.mbits);
  rs.kstar = 0u;
  rs.keep = 0;
  rs.total = 0;
  rs.tie_cut = V;
  rs.all_kept = filt ? 0 : 1;
  DF z = sh.z;
  double zfull = df_double(z);
  const bool bad = bad_t || !isfinite(rs.m) || !(fabsf(rs.m * c) < 1073741824.f);
  rs.bad = bad ? 1 : 0;
  double zk = zfull;
  int nlist = 0;
  bool from_list = false;
  if (filt && !bad) {
    bool done = false;
    if (hist_on && !sh.corrupt && isfinite(zfull) && zfull > 0.0) {
      done = cut_from_hist<DT>(sh, reinterpret_cast<const uint32_t*>(dsm), rs, a.top_k, a.top_p, zfull, sh.kb, &zk);
      nlist = sh.nlist;
      from_list = done && nlist <= kListCap;
    }
    if (!done) {
      if (!(isfinite(zfull) && zfull > 0.0)) zfull = row_pass<DT>(sh, row, V, aligned, PASS_MASS_GT, 0u, rs);
      const CutOut co = search_cut<DT>(sh, row, V, aligned, a.top_k, a.top_p, rs, zfull);
      rs.kstar = co.kstar;
      rs.keep = static_cast<int>(co.keep);
      rs.total = static_cast<int>(co.total);
      zk = df_double(co.zkept);
    }
    if (rs.keep < rs.total) {
      rs.tie_cut = from_list ? tie_cut_from_list<DT>(sh, dsm, reinterpret_cast<uint32_t*>(dsm), nlist, rs.kstar,
                                                      rs.keep, rs.total)
                             : -1;
      // rows that searched the whole row find the bound now; rows whose
      // candidate list overflowed leave it to whoever needs it
      if (rs.tie_cut < 0 && (!hist_on || !done || role == ROLE_PROBS)) {
        const int idx = find_nth_equal<DT>(sh, row, V, aligned, 0, nvec, rs.kstar, rs.keep);
        rs.tie_cut = idx < 0 ? V : idx + 1;
      }
    }
  } else if (!bad && !(isfinite(zfull) && zfull > 0.0)) {
    zfull = row_pass<DT>(sh, row, V, aligned, PASS_MASS_GT, 0u, rs);
    zk = zfull;
  }
  rs.zkept = static_cast<float>(zk);
  rs.inv_z = static_cast<float>(1.0 / zk);

  if (role == ROLE_PROBS) {
    float* out = a.out_probs + static_cast<size_t>(item) * V;
    if (bad) {
      for (int t = tid; t < V; t += kThreads) out[t] = 0.f;
      if (tid == 0) set_status(a.status, SPEC_STATUS_BAD_ROW);
    } else {
      write_probs<DT>(row, V, aligned, rs, out);
    }
    return;
  }

  // the probability at the draft token (its rank among ties found by a pass
  // over the row before it when the bound is not known)
  bool xkept = false;
  float xp = 0.f;
  if (paired && xok && !bad) {
    const uint32_t xk = E::key(sh.xbits);
    if (rs.all_kept || xk > rs.kstar) xkept = true;
    else if (xk == rs.kstar) {
      if (rs.tie_cut >= 0) xkept = xtok < rs.tie_cut;
      else xkept = count_equal<DT>(sh, row, V, aligned, 0, xtok / E::kPerVec + 1, rs.kstar, xtok) <
                   static_cast<uint32_t>(rs.keep);
    }
    if (xkept) xp = lat_mass(E::value(sh.xbits), rs.c, rs.K) * rs.inv_z;
  }

  // ------------------------------------------------------------- publish
  RowPub* const pub = a.pubs + rr.pub;
  if (role == ROLE_P || role == ROLE_BONUS) {
    uint32_t nl = kPubReread;
    if (from_list && !bad && rs.tie_cut >= 0) {
      const int nkv = kept_vectors<DT>(sh, dsm, nlist, nvec, rs.kstar, pub->list);
      if (nkv <= kPubList) nl = static_cast<uint32_t>(nkv);
    }
    if (tid == 0) pub->nlist = nl;
  }
  if (tid == 0) {
    pub->rs = rs;
    pub->xprob = xp;
    if (role == ROLE_P && a.out_p) a.out_p[static_cast<size_t>(b) * a.k + pos] = xp;
    if (role == ROLE_Q && a.out_q) a.out_q[static_cast<size_t>(b) * a.k + pos] = xp;
    const uint32_t st = (bad ? SPEC_STATUS_BAD_ROW : 0u) | ((role == ROLE_P && !xok) ? SPEC_STATUS_BAD_TOKEN : 0u);
    if (st) set_status(a.status, st);
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    sh.second = atomicAdd(a.seq_tickets + b, 1u) == static_cast<uint32_t>(2 * a.k) ? 1 : 0;
  }
  __syncthreads();
  if (sh.second) finish_sequence<DT>(a, sh, dsm, b);
}

// ----------------------------------------------------- whole-row draws
// Queue entry e (sequence b, first rejection n) is drawn in a.chunks chunks
// of the rows' vectors, one CTA each: (1) rows whose tie bound is not known
// count their tokens of value kstar per chunk; (2) each chunk, knowing how
// many such tokens come before it, sets its own bound and sums its draw
// weights; the last chunk to finish picks the chunk holding u * S and walks
// it.
struct DrawRows {
  int n;
  bool want_q, bad, need_p, need_q;
  RowStat rp, rq;
  const unsigned char *rowp, *rowq;
  bool ap, aq;
};
template <int DT>
__device__ __forceinline__ DrawRows draw_rows(const SampleArgs& a, int b) {
  using E = Elt<DT>;
  DrawRows d;
  const int k = a.k;
  d.n = min(max(__ldcg(a.out_n + b), 0), k);
  d.want_q = d.n < k;
  const RowPub* const pp =
      d.want_q ? a.pubs + 2 * (static_cast<size_t>(b) * k + d.n) : a.pubs + 2 * static_cast<size_t>(a.B) * k + b;
  d.rp = ldcg_rowstat(&pp[0].rs);
  d.rq = d.want_q ? ldcg_rowstat(&pp[1].rs) : d.rp;
  d.bad = d.rp.bad || (d.want_q && d.rq.bad);
  d.need_p = !d.rp.all_kept && d.rp.tie_cut < 0;
  d.need_q = d.want_q && !d.rq.all_kept && d.rq.tie_cut < 0;
  const size_t rb = static_cast<size_t>(a.V) * E::kBytes;
  d.rowp = static_cast<const unsigned char*>(a.target) + (static_cast<size_t>(b) * (k + 1) + d.n) * rb;
  d.rowq = d.want_q ? static_cast<const unsigned char*>(a.draft) + (static_cast<size_t>(b) * k + d.n) * rb : d.rowp;
  d.ap = a.aligned_target != 0;
  d.aq = d.want_q ? a.aligned_draft != 0 : d.ap;
  return d;
}
__device__ __forceinline__ int chunk_beg(int nvec, int S, int cc) {
  return static_cast<int>(static_cast<long long>(nvec) * cc / S);
}

// Stage 1: tokens of value kstar in chunk s (rows whose bound is unknown).
template <int DT>
__device__ __noinline__ void draw_count(const SampleArgs& a, Shm& sh, int b, int s) {
  using E = Elt<DT>;
  const DrawRows d = draw_rows<DT>(a, b);
  if (d.bad || !(d.need_p || d.need_q)) return;
  const int nvec = (a.V + E::kPerVec - 1) / E::kPerVec, S = a.chunks;
  const int e0 = chunk_beg(nvec, S, s), e1 = chunk_beg(nvec, S, s + 1);
  const uint32_t cp = d.need_p ? count_equal<DT>(sh, d.rowp, a.V, d.ap, e0, e1, d.rp.kstar, a.V) : 0u;
  const uint32_t cq = d.need_q ? count_equal<DT>(sh, d.rowq, a.V, d.aq, e0, e1, d.rq.kstar, a.V) : 0u;
  if (threadIdx.x == 0) {
    int32_t* t = a.tcnt + (static_cast<size_t>(b) * kMaxDrawChunks + s) * 2;
    t[0] = static_cast<int32_t>(cp);
    t[1] = static_cast<int32_t>(cq);
    __threadfence();
    atomicAdd(a.tie_tickets + b, 1u);
  }
}
template <int DT>
__device__ __forceinline__ bool draw_needs_counts(const SampleArgs& a, int b) {
  const DrawRows d = draw_rows<DT>(a, b);
  return !d.bad && (d.need_p || d.need_q);
}

// The bound of one row's tie inside chunk s, from the per-chunk counts.
template <int DT>
__device__ __forceinline__ int chunk_tie_cut(const SampleArgs& a, Shm& sh, int b, int s, int which, const RowStat& r,
                                             const unsigned char* row, bool al, int e0, int e1) {
  int before = 0;
  for (int cc = 0; cc < s; ++cc) before += __ldcg(a.tcnt + (static_cast<size_t>(b) * kMaxDrawChunks + cc) * 2 + which);
  const int mine = __ldcg(a.tcnt + (static_cast<size_t>(b) * kMaxDrawChunks + s) * 2 + which);
  if (before + mine <= r.keep) return 0x7FFFFFFF;  // every such token of this chunk is kept
  if (before >= r.keep) return 0;                  // none is
  const int idx = find_nth_equal<DT>(sh, row, a.V, al, e0, e1, r.kstar, r.keep - before);
  return idx < 0 ? 0 : idx + 1;
}

// Stage 2 of chunk s; the last chunk picks and walks.  e: the queue entry.
template <int DT>
__device__ __noinline__ void draw_sum(const SampleArgs& a, Shm& sh, int b, int s, int e) {
  using E = Elt<DT>;
  const int tid = threadIdx.x, S = a.chunks, k = a.k;
  DrawRows d = draw_rows<DT>(a, b);
  const int nvec = (a.V + E::kPerVec - 1) / E::kPerVec;
  const int e0 = chunk_beg(nvec, S, s), e1 = chunk_beg(nvec, S, s + 1);
  const float u = a.uniforms[static_cast<size_t>(b) * (k + 2) + (d.want_q ? k + 1 : k)];
  RowStat rp = d.rp, rq = d.rq;
  if (!d.bad) {
    __threadfence();
    if (d.need_p) rp.tie_cut = chunk_tie_cut<DT>(a, sh, b, s, 0, d.rp, d.rowp, d.ap, e0, e1);
    if (d.need_q) rq.tie_cut = chunk_tie_cut<DT>(a, sh, b, s, 1, d.rq, d.rowq, d.aq, e0, e1);
    if (tid == 0) {
      int32_t* t = a.tcut + (static_cast<size_t>(b) * kMaxDrawChunks + s) * 2;
      t[0] = rp.tie_cut;
      t[1] = rq.tie_cut;
    }
    range_sums<DT>(sh, rp, rq, d.rowp, d.rowq, d.ap, d.aq, a.V, d.want_q, nullptr, e0, e1);
  } else {
    if (tid < kWarps) {
      sh.w_s[tid] = 0.f;
      sh.w_sp[tid] = 0.f;
    }
    __syncthreads();
  }
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
    for (int w = 0; w < kWarps; ++w) {
      cs[4 + w] = sh.w_s[w];
      cs[4 + kWarps + w] = sh.w_sp[w];
    }
    __threadfence();
    sh.second = atomicAdd(a.draw_tickets + b, 1u) == static_cast<uint32_t>(S - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!sh.second) return;

  // ---------------------------------------- the last chunk: pick one, walk it
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
    const bool use_q = d.want_q && tr.hi > 0.f;  // a residual with no mass: draw from p
    const DF target = df_mul_f(use_q ? tr : tp, u);
    DF run{0.f, 0.f}, base{0.f, 0.f}, lbase{0.f, 0.f};
    int csel = -1, clast = -1;
    const int o = use_q ? 0 : 2;
    for (int cc = 0; cc < S; ++cc) {
      const DF sc{cs[4 * cc + o], cs[4 * cc + o + 1]};
      const DF nx = df_add2(run, sc);
      if (sc.hi > 0.f) {
        clast = cc;
        lbase = run;
      }
      if (csel < 0 && sc.hi > 0.f && df_lt(target, nx)) {
        csel = cc;
        base = run;
      }
      run = nx;
    }
    if (csel < 0) {
      csel = clast;
      base = lbase;
    }
    sh.draw_chunk = d.bad ? -1 : csel;
    sh.draw_useq = use_q ? 1 : 0;
    sh.draw_target = df_add2(target, df_neg(base));
  }
  __syncthreads();
  const int cs = sh.draw_chunk;
  int token = -1;
  if (cs >= 0) {
    const bool use_q = sh.draw_useq != 0;
    if (tid < 2 * kWarps) {
      const float v = __ldcg(a.csums + (static_cast<size_t>(b) * kMaxDrawChunks + cs) * kChunkRec + 4 + tid);
      if (tid < kWarps) sh.w_s[tid] = v;
      else sh.w_sp[tid - kWarps] = v;
    }
    RowStat wp = d.rp, wq = d.rq;
    if (d.need_p) wp.tie_cut = __ldcg(a.tcut + (static_cast<size_t>(b) * kMaxDrawChunks + cs) * 2);
    if (d.need_q) wq.tie_cut = __ldcg(a.tcut + (static_cast<size_t>(b) * kMaxDrawChunks + cs) * 2 + 1);
    __syncthreads();
    token = range_walk<DT>(sh, wp, wq, d.rowp, d.rowq, d.ap, d.aq, a.V, use_q, sh.draw_target, nullptr,
                           chunk_beg(nvec, S, cs), chunk_beg(nvec, S, cs + 1));
  }
  if (tid == 0) {
    a.out_tokens[static_cast<size_t>(b) * (k + 1) + d.n] = token;
    // left zeroed for the next call
    a.draw_tickets[b] = 0u;
    a.tie_tickets[b] = 0u;
    a.ready[e] = 0u;
  }
  clear_sequence(a, b, true);
}

}  // namespace

// ------------------------------------------------------------------ kernels
// One row per CTA (the separate-launch mode).
template <int DT>
__global__ void __launch_bounds__(kThreads, 4) rows_kernel(const SampleArgs a) {
  __shared__ Shm sh;
  extern __shared__ __align__(16) unsigned char dsm[];
  process_row<DT>(a, sh, dsm, static_cast<int>(blockIdx.x));
}
// Whole-row draws, separate-launch mode: counts, then sums and walks.
template <int DT>
__global__ void __launch_bounds__(kThreads, 4) draw1_kernel(const SampleArgs a) {
  __shared__ Shm sh;
  const int e = static_cast<int>(blockIdx.x) / a.chunks, s = static_cast<int>(blockIdx.x) % a.chunks;
  if (e >= static_cast<int>(__ldcg(a.work + WK_QUEUED))) return;
  const int b = static_cast<int>(__ldcg(a.ready + e)) - 1;
  if (b < 0) return;
  draw_count<DT>(a, sh, b, s);
}
template <int DT>
__global__ void __launch_bounds__(kThreads, 4) draw2_kernel(const SampleArgs a) {
  __shared__ Shm sh;
  const int e = static_cast<int>(blockIdx.x) / a.chunks, s = static_cast<int>(blockIdx.x) % a.chunks;
  if (e < static_cast<int>(__ldcg(a.work + WK_QUEUED))) {
    const int b = static_cast<int>(__ldcg(a.ready + e)) - 1;
    if (b >= 0) draw_sum<DT>(a, sh, b, s, e);
  }
  // the last CTA out leaves the counters zeroed for the next call
  __syncthreads();
  if (threadIdx.x == 0 && atomicAdd(a.work + WK_EXIT, 1u) == gridDim.x - 1) {
    a.work[WK_QUEUED] = 0u;
    a.work[WK_SEQS] = 0u;
    a.work[WK_EXIT] = 0u;
  }
}
// Separate-launch mode of spec_transform_probs and of sampling calls with
// no whole-row draw to run: the counters the finishers bump are reset here.
__global__ void reset_kernel(uint32_t* work) {
  if (threadIdx.x < 8) work[threadIdx.x] = 0u;
}

// One cooperative launch of as many CTAs as fit on the GPU, taking work items
// in order from counters: every row, then the whole-row draw chunks.  A draw
// chunk waits (bounded polls) for its queue entry and, when ties must be
// counted, for the other chunks of its entry to count theirs; the awaited
// work was taken earlier by running CTAs and waits on nothing it could block,
// so every wait ends.  Past the poll limit the wait gives up and sets
// SPEC_STATUS_TIMEOUT (that token stays -1).
template <int DT>
__global__ void __launch_bounds__(kThreads, 4) fused_kernel(const SampleArgs a) {
  __shared__ Shm sh;
  extern __shared__ __align__(16) unsigned char dsm[];
  const int R = a.mode == MODE_SAMPLE ? a.B * (2 * a.k + 1) : a.B;
  const int tid = threadIdx.x;
  for (;;) {
    __syncthreads();
    if (tid == 0) sh.item = static_cast<int>(atomicAdd(a.work + WK_ROWS, 1u));
    __syncthreads();
    const int item = sh.item;
    if (item >= R) break;
    process_row<DT>(a, sh, dsm, item);
  }
  if (a.mode == MODE_SAMPLE) {
    const int S = a.chunks;
    for (;;) {
      __syncthreads();
      if (tid == 0) {
        const int d = static_cast<int>(atomicAdd(a.work + WK_DRAWS, 1u));
        const int e = d / S;
        int bb = -2;  // -2: no more queued draws; -1: the wait gave up
        if (e < a.B) {
          bb = -1;
          for (int i = 0; i < a.poll_limit; ++i) {
            const uint32_t v = ld_acquire_u32(a.ready + e);
            if (v) {
              bb = static_cast<int>(v) - 1;
              break;
            }
            if (ld_acquire_u32(a.work + WK_SEQS) == static_cast<uint32_t>(a.B) &&
                ld_acquire_u32(a.work + WK_QUEUED) <= static_cast<uint32_t>(e)) {
              bb = -2;
              break;
            }
            __nanosleep(64);
          }
          if (bb == -1) set_status(a.status, SPEC_STATUS_TIMEOUT);
        }
        sh.item = d;
        sh.flag = bb;
      }
      __syncthreads();
      const int bb = sh.flag;
      if (bb == -2) break;
      if (bb < 0) continue;
      const int e = sh.item / S, s = sh.item % S;
      if (draw_needs_counts<DT>(a, bb)) {
        draw_count<DT>(a, sh, bb, s);
        if (tid == 0) {
          int ok = 0;
          for (int i = 0; i < a.poll_limit; ++i) {
            if (ld_acquire_u32(a.tie_tickets + bb) >= static_cast<uint32_t>(S)) {
              ok = 1;
              break;
            }
            __nanosleep(64);
          }
          if (!ok) set_status(a.status, SPEC_STATUS_TIMEOUT);
          sh.flag = ok;
        }
        __syncthreads();
        if (!sh.flag) continue;
      }
      draw_sum<DT>(a, sh, bb, s, e);
    }
  }
  // the last CTA out leaves the counters zeroed for the next call
  __syncthreads();
  if (tid == 0 && atomicAdd(a.work + WK_EXIT, 1u) == gridDim.x - 1) {
    for (int i = 0; i < 8; ++i) a.work[i] = 0u;
  }
}

// ------------------------------------------------------------------ launch

size_t sample_smem_bytes(int dtype, bool filter) {
  return (dtype == DT_BF16 && filter) ? kRowSmem : sizeof(uint32_t) * 3 * kPubList;
}

template <int DT>
static int launch_all(const SampleArgs& args, cudaStream_t st) {
  SampleArgs a = args;
  a.poll_limit = a.launch_mode == SPEC_LAUNCH_FUSED_WAIT_TEST ? 64 : kMaxPolls;
  const bool filter = a.top_k > 0 || a.top_p < 1.f;
  const int rows = a.mode == MODE_SAMPLE ? a.B * (2 * a.k + 1) : a.B;
  const size_t smem = sample_smem_bytes(DT, filter);
  bool fused = false;
  if (a.launch_mode != SPEC_LAUNCH_SEPARATE) {
    int per_sm = 0, dev = 0, coop = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
        cudaFuncSetAttribute(fused_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) ==
            cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_kernel<DT>, kThreads, smem) == cudaSuccess &&
        per_sm > 0) {
      const int items = rows + (a.mode == MODE_SAMPLE ? a.B * a.chunks : 0);
      const int grid = std::min(per_sm * num_sms(), items);
      void* params[] = {&a};
      fused = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fused_kernel<DT>), dim3(grid), dim3(kThreads),
                                          params, smem, st) == cudaSuccess;
    }
    if (!fused) (void)cudaGetLastError();  // (clear a refused launch; the separate launches stand in)
  }
  if (!fused) {
    cudaFuncSetAttribute(rows_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    rows_kernel<DT><<<rows, kThreads, smem, st>>>(a);
    if (a.mode == MODE_SAMPLE) {
      draw1_kernel<DT><<<a.B * a.chunks, kThreads, 0, st>>>(a);
      draw2_kernel<DT><<<a.B * a.chunks, kThreads, 0, st>>>(a);
    } else {
      reset_kernel<<<1, 32, 0, st>>>(a.work);
    }
  }
  return cudaGetLastError();
}

int launch_sample(const SampleArgs& a, int dtype, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == DT_BF16) return launch_all<DT_BF16>(a, st);
  if (dtype == DT_F32) return launch_all<DT_F32>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace specv
