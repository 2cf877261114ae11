// split_kernel.cu -- speculative-sampling verification as three launches:
// stream, row, draw.
//
// The method (Edge Inference Notes, post on speculative decoding and EAGLE-3,
// "The core idea: draft, then check", step 3; temperature, top-k and nucleus
// applied to both distributions as "Why it changes nothing about the output"
// states): for positions i = 0..k-1 the draft token x_i is accepted iff
// u_i q_i(x_i) < p_i(x_i); at the first rejection n one token is drawn from
// max(0, p_n - q_n) (renormalised) with u_{k+1}; if every draft is accepted
// the bonus token is drawn from p_k with u_k.
//
// Design.  Every row is read from HBM once, by a kernel that does nothing
// but stream; what the filters need is gathered on the way, so that deciding
// a row afterwards reads a few KB.
//   stream  The target rows, then the draft rows, laid end to end as 16-byte
//           vectors and cut into one equal range per CTA (one wave).  Per
//           row piece every warp keeps its running maximum, its mass sum
//           2^((v - m) c) (c = log2(e)/T) and, with a filter, exact counts
//           of the bf16 keys in a window below its running maximum: at most
//           kSW keys and kBandOct octaves of mass (a ring indexed by key mod
//           kSW, cleared as the maximum rises).  The vectors holding such
//           values are listed in shared memory and counted 32 at a time.
//           Counts of tokens before the position's draft token and from it
//           on are kept apart.  A piece leaves a record: its maximum, its
//           mass and the counts below its own maximum key.
//   row     One CTA per row merges the records of the row's pieces: the
//           maximum, Z, and the window counts of the row.  The cut of top-k
//           (a count) and top-p (a mass, over the top-k set) is the group of
//           equal values where the running total over the window, from the
//           top, reaches its target; the lowest indices of that group are
//           kept.  The draft token's rank within its group comes from the
//           counts before it.  Rows whose cut lies below the window are
//           searched in their own row, one window of kSW keys per pass,
//           downwards.  Each row leaves p(x) (or q(x)) and
//           its kept set as (cut key, tokens of that key kept, kept mass).
//   draw    One cluster of kDrawCl CTAs per sequence finds n from the rows'
//           p(x), q(x) and u, commits the accepted drafts and draws at n:
//           every CTA takes a slice of the row pair, ranks the cut group's
//           tokens by index across the cluster (distributed shared memory),
//           sums max(0, p - q) per warp, and the CTA holding u S walks to the
//           token.
// Sums over elements are float per thread and double-float (two floats)
// above; no double precision is used.  The filters need bf16 rows (exact
// 16-bit keys); f32 rows take this path only without a filter.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"

namespace specv {
namespace {

constexpr int kSW = 512;             // window keys per piece
constexpr int kSUnroll = 8;          // 16-byte loads in flight per thread (stream)
constexpr int kList = 32 + 32 * kSUnroll;  // candidate vectors a warp lists between countings (stream)
constexpr int kDrawCl = 16;          // CTAs per sequence (draw; a non-portable cluster size)
constexpr int kDrawThreads = 128;    // threads per draw CTA
constexpr int kDrawWarps = kDrawThreads / 32;
constexpr unsigned kFullMask = 0xFFFFFFFFu;
constexpr int kMaxPiecesPerRow = 64;
constexpr float kBandOct = 16.f;     // counted values carry at least 2^-16 of the maximum's mass

// One row piece after the stream kernel (in the workspace's tag area, slot
// cta + row).
struct PieceRec {
  float m;              // maximum of the piece (-inf: no finite entry)
  float zh, zl;         // sum of 2^((v - m) c) over the piece, double-float
  uint32_t top;         // key of m
  uint32_t nan;         // a NaN or +inf was seen
  uint32_t pad[3];
  uint32_t hist[kSW];   // hist[j]: tokens of key top - j
};
static_assert(sizeof(PieceRec) % 16 == 0, "records stay 16-byte aligned");

// One row after the row kernel (in the row's RowHdr slot).
struct SRow {
  float m;              // row maximum
  float c;              // log2(e) / T
  float izk;            // 1 / kept mass
  uint32_t kstar;       // cut key (every key above it is kept)
  int32_t keep;         // tokens of key kstar kept: the lowest indices
  int32_t gcount;       // tokens of key kstar in the row
  int32_t all_kept;     // no filter, or the filter keeps every token
  int32_t bad;          // non-finite row or temperature
  float xprob;          // p(x) (target rows) or q(x) (draft rows) at the position's draft token
  float zkh, zkl;       // kept mass, double-float
  int32_t pad[5];
};
static_assert(sizeof(SRow) <= sizeof(RowHdr), "a row's outcome lives in its header slot");

// ------------------------------------------------------------ double-float

struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF df_make(float x) { return DF{x, 0.f}; }
__device__ __forceinline__ DF df_add(DF a, float x) {  // TwoSum
  const float s = a.hi + x;
  const float bp = s - a.hi;
  const float e = (a.hi - (s - bp)) + (x - bp);
  return DF{s, a.lo + e};
}
__device__ __forceinline__ DF df_add(DF a, DF b) {
  DF r = df_add(a, b.hi);
  r.lo += b.lo;
  return r;
}
__device__ __forceinline__ DF df_norm(DF a) {
  const float s = a.hi + a.lo;
  return DF{s, a.lo - (s - a.hi)};
}
__device__ __forceinline__ DF df_neg(DF a) { return DF{-a.hi, -a.lo}; }
__device__ __forceinline__ DF df_mulf(DF a, float f) {
  const float p = a.hi * f;
  const float e = fmaf(a.hi, f, -p);
  return df_norm(DF{p, fmaf(a.lo, f, e)});
}
__device__ __forceinline__ bool df_lt(DF a, DF b) { return df_norm(df_add(a, df_neg(b))).hi < 0.f; }
__device__ __forceinline__ float df_f(DF a) { return a.hi + a.lo; }
__device__ __forceinline__ DF shfl_df(DF a, int src) {
  return DF{__shfl_sync(kFullMask, a.hi, src), __shfl_sync(kFullMask, a.lo, src)};
}
__device__ __forceinline__ DF shfl_up_df(DF a, int d) {
  return DF{__shfl_up_sync(kFullMask, a.hi, d), __shfl_up_sync(kFullMask, a.lo, d)};
}
__device__ __forceinline__ DF warp_sum_df(DF a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = df_add(a, DF{__shfl_xor_sync(kFullMask, a.hi, o), __shfl_xor_sync(kFullMask, a.lo, o)});
  return df_norm(a);
}
__device__ __forceinline__ DF warp_incl_scan_df(DF a) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF b = shfl_up_df(a, o);
    if (lane >= o) a = df_add(a, b);
  }
  return df_norm(a);
}

// ------------------------------------------------------------ small helpers

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(kFullMask, v, o));
  return v;
}
__device__ __forceinline__ uint32_t warp_incl_scan_u(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFullMask, v, o);
    if (lane >= o) v += y;
  }
  return v;
}
__device__ __forceinline__ float mass(float v, float c, float nmc) { return ex2_approx(fmaf(v, c, nmc)); }
// Packed pairs of floats (f32x2 arithmetic, per element the same fma as mass()).
typedef unsigned long long u64;
__device__ __forceinline__ u64 pk2(uint32_t x, uint32_t y) {
  u64 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(x), "r"(y));
  return r;
}
__device__ __forceinline__ void upk2(u64 r, float& x, float& y) { asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(r)); }
__device__ __forceinline__ u64 fma_x2(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ u64 add_x2(u64 a, u64 b) {
  u64 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Masses of the two bf16 values of one 32-bit word, added into acc.
__device__ __forceinline__ u64 mass_word(uint32_t wd, u64 c2, u64 n2, u64 acc) {
  float e0, e1;
  upk2(fma_x2(pk2(wd << 16, wd & 0xFFFF0000u), c2, n2), e0, e1);
  return add_x2(acc, pk2(__float_as_uint(ex2_approx(e0)), __float_as_uint(ex2_approx(e1))));
}
__device__ __forceinline__ uint32_t bkey(uint32_t bits) { return Elt<DT_BF16>::key(bits); }
__device__ __forceinline__ float bval_of_key(uint32_t key) { return Elt<DT_BF16>::value(Elt<DT_BF16>::bits_of_key(key)); }
// bf16 bits of a value threshold for "key >= kl" on non-NaN values (keys below
// that of -inf are NaN patterns: everything non-NaN is above them)
__device__ __forceinline__ uint32_t floor_bits2(uint32_t kl) {
  const uint32_t b = kl <= 0x7Fu ? 0xFF80u : Elt<DT_BF16>::bits_of_key(kl);
  return b | (b << 16);
}
// Lowest key counted below a maximum m (of key pm): within kSW keys of it and
// within kBandOct octaves of mass (values >= m - kBandOct / c; the largest bf16
// value not above that bound).  The stream and row kernels compute it alike.
__device__ __forceinline__ uint32_t band_floor(float m, uint32_t pm, float c) {
  uint32_t f = pm >= static_cast<uint32_t>(kSW - 1) ? pm - static_cast<uint32_t>(kSW - 1) : 0u;
  if (c > 0.f) {
    const float vf = m - kBandOct / c;
    if (vf > -INFINITY) {
      const uint32_t u = __float_as_uint(vf);
      uint32_t hi = u >> 16;
      if ((u & 0xFFFFu) != 0u && (u & 0x80000000u) != 0u) hi += 1u;  // negative: one step further down
      f = max(f, bkey(hi));
    }
  }
  return f;
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
  return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}

// ------------------------------------------------------------ row geometry

// Rows of a call: the B(k+1) target rows, then the Bk draft rows.
struct RowRef {
  const unsigned char* ptr;
  int b, i;
  bool target;
  int x;  // the position's draft token, -1 for the bonus row or a token outside [0, V)
};
__device__ __forceinline__ RowRef row_ref(const SampleArgs& a, int r, int ebytes) {
  RowRef rr;
  const int rt = a.B * (a.k + 1);
  const size_t rb = static_cast<size_t>(a.V) * ebytes;
  if (r < rt) {
    rr.b = r / (a.k + 1);
    rr.i = r % (a.k + 1);
    rr.target = true;
    rr.ptr = static_cast<const unsigned char*>(a.target) + static_cast<size_t>(r) * rb;
  } else {
    const int d = r - rt;
    rr.b = d / a.k;
    rr.i = d % a.k;
    rr.target = false;
    rr.ptr = static_cast<const unsigned char*>(a.draft) + static_cast<size_t>(d) * rb;
  }
  rr.x = -1;
  if (rr.i < a.k) {
    const int x = a.tokens[static_cast<size_t>(rr.b) * a.k + rr.i];
    if (x >= 0 && x < a.V) rr.x = x;
  }
  return rr;
}
__device__ __forceinline__ float row_c(const SampleArgs& a, int b) {
  const float T = a.temperature_per_seq ? a.temperature_per_seq[b] : a.temperature;
  return (T > 0.f && isfinite(T)) ? kLog2e / T : 0.f;
}
// Equal ranges of the stream grid: the first vector of CTA g.
__device__ __forceinline__ long long range_start(long long units, int grid, long long g) { return g * units / grid; }
// The CTA whose range holds vector u.
__device__ __forceinline__ int cta_of(long long units, int grid, long long u) {
  return static_cast<int>(((u + 1) * grid - 1) / units);
}
__device__ __forceinline__ PieceRec* piece_rec(const SampleArgs& a, int cta, int row) {
  return reinterpret_cast<PieceRec*>(a.tags) + (static_cast<size_t>(cta) + row);
}
// Counts before the draft token, written by the piece that holds it.
__device__ __forceinline__ uint32_t* before_hist(const SampleArgs& a, int row) { return a.pubs[row].list; }

// Counts a warp's listed candidate vectors: every value at or above fv into
// the warp's window (slot key mod kSW, two 16-bit counts a word; tokens
// before x in the first half of the window, from x on in the second).  A
// warp's share of one row stays below 2^16 tokens (rows of at most 2^18).
__device__ __forceinline__ void count_list(const uint4* wl, const int* wi, int nl, uint32_t* wh, int x, float fv) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < nl; e += 32) {
    const uint4 vq = wl[e];
    const int vi = wi[e];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t wd = word_of(vq, j >> 1);
      const uint32_t bits = (j & 1) ? (wd >> 16) : (wd & 0xFFFFu);
      if (__uint_as_float(bits << 16) >= fv) {
        const uint32_t sl = bkey(bits) & static_cast<uint32_t>(kSW - 1);
        const int idx = vi * 8 + j;
        red_add_shared(smem_addr(wh + (idx >= x ? kSW / 2 : 0) + (sl >> 1)), 1u << (16u * (sl & 1u)));
      }
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------ stream kernel

// One wave of CTAs over every row of the call (target rows, then draft rows),
// each CTA an equal range of 16-byte vectors; see the file comment.
template <int DT, bool HIST>
__global__ void __launch_bounds__(kThreads, 4) split_stream_kernel(const SampleArgs a) {
  using E = Elt<DT>;
  constexpr int PV = E::kPerVec;
  static_assert(!HIST || DT == DT_BF16, "window counts need bf16 keys");
  // per warp: counts of the window's keys (key mod kSW), two 16-bit counts a
  // word, tokens before x in the first half and from x on in the second
  __shared__ __align__(16) uint32_t hist[HIST ? kWarps * kSW : 1];
  __shared__ __align__(16) uint4 lst[HIST ? kWarps * kList : 1];  // candidate vectors, then their indices
  __shared__ int lidx[HIST ? kWarps * kList : 1];
  __shared__ float s_m[kWarps];
  __shared__ uint32_t s_nan[kWarps], s_top[kWarps], s_floor[kWarps];
  __shared__ DF s_z[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.B * (2 * a.k + 1);
  const long long nvr = a.V / PV;
  const long long units = static_cast<long long>(R) * nvr;
  const int grid = static_cast<int>(gridDim.x);
  const long long u0 = range_start(units, grid, blockIdx.x), u1 = range_start(units, grid, blockIdx.x + 1);
  uint32_t* const wh = hist + (HIST ? warp * kSW : 0);
  uint4* const wl = lst + (HIST ? warp * kList : 0);
  int* const wi = lidx + (HIST ? warp * kList : 0);
  constexpr uint32_t kPadWord = DT == DT_BF16 ? 0xFF80FF80u : 0xFF800000u;  // -inf

  for (long long us = u0; us < u1;) {
    const int row = static_cast<int>(us / nvr);
    const long long rbeg = static_cast<long long>(row) * nvr;
    const long long ue = min(u1, rbeg + nvr);
    const int v_lo = static_cast<int>(us - rbeg), v_hi = static_cast<int>(ue - rbeg);
    us = ue;
    const RowRef rr = row_ref(a, row, E::kBytes);
    const float c = row_c(a, rr.b);
    const int x = rr.x;  // counts of tokens before x and from x on are kept apart
    if (HIST) {
      for (int j = lane; j < kSW; j += 32) wh[j] = 0u;
      __syncwarp();
    }
    int nl = 0;  // candidate vectors listed by this warp (warp-uniform)
    // warp-uniform: running maximum, its key (window top), window floor key
    float Mw = -INFINITY, nmc = 0.f;
    uint32_t Pw = 0u, Fw = 0u, t2 = 0u, nanw = 0u;
    DF z = df_make(0.f);
    const uint4* const vp = reinterpret_cast<const uint4*>(rr.ptr);
    for (int base = v_lo; base < v_hi; base += kThreads * kSUnroll) {
      uint4 q[kSUnroll];
#pragma unroll
      for (int u = 0; u < kSUnroll; ++u) {
        const int v = base + u * kThreads + tid;
        q[u] = v < v_hi ? ldg_stream(vp + v) : make_uint4(kPadWord, kPadWord, kPadWord, kPadWord);
      }
      float tm;
      if constexpr (DT == DT_BF16) {
        uint32_t m2 = 0xFF80FF80u;
#pragma unroll
        for (int u = 0; u < kSUnroll; ++u)
          m2 = bmax2_nan(m2, bmax2_nan(bmax2_nan(q[u].x, q[u].y), bmax2_nan(q[u].z, q[u].w)));
        tm = max_nan(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
      } else {
        tm = -INFINITY;
#pragma unroll
        for (int u = 0; u < kSUnroll; ++u)
          tm = max_nan(tm, max_nan(max_nan(__uint_as_float(q[u].x), __uint_as_float(q[u].y)),
                                   max_nan(__uint_as_float(q[u].z), __uint_as_float(q[u].w))));
      }
      const float wm = warp_max_nan(tm);
      if (wm != wm || wm == INFINITY) {
        nanw = 1u;
      } else if (wm > Mw) {  // a new running maximum: rescale, slide the window
        if (Mw > -INFINITY) z = df_mulf(z, ex2_approx((Mw - wm) * c));
        if constexpr (HIST) {
          const uint32_t Pn = bkey(__float_as_uint(wm) >> 16);
          const uint32_t Fn = band_floor(wm, Pn, c);
          if (Mw > -INFINITY && Fn > Fw) {  // the keys that left the window free their slots
            if (Fn - Fw >= static_cast<uint32_t>(kSW)) {
              for (int j = lane; j < kSW; j += 32) wh[j] = 0u;
            } else {
              for (int w2 = lane; w2 < kSW / 2; w2 += 32) {  // (a word holds slots 2 w2 and 2 w2 + 1)
                uint32_t keep = 0u;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const uint32_t sl = 2u * static_cast<uint32_t>(w2) + h;
                  const uint32_t d = (sl - Fw) & static_cast<uint32_t>(kSW - 1);  // slot of key Fw + d
                  if (d >= Fn - Fw) keep |= 0xFFFFu << (16 * h);
                }
                if (keep != 0xFFFFFFFFu) {
                  wh[w2] &= keep;
                  wh[kSW / 2 + w2] &= keep;
                }
              }
            }
            __syncwarp();
          }
          Pw = Pn;
          Fw = Fn;
          t2 = floor_bits2(Fn);
        }
        Mw = wm;
        nmc = -wm * c;
      }
      if (nanw || !(Mw > -INFINITY)) continue;
      if constexpr (DT == DT_BF16) {
        const u64 c2 = pk2(__float_as_uint(c), __float_as_uint(c)), n2 = pk2(__float_as_uint(nmc), __float_as_uint(nmc));
        u64 acc = pk2(0u, 0u);
#pragma unroll
        for (int u = 0; u < kSUnroll; ++u) {
          acc = mass_word(q[u].x, c2, n2, acc);
          acc = mass_word(q[u].y, c2, n2, acc);
          acc = mass_word(q[u].z, c2, n2, acc);
          acc = mass_word(q[u].w, c2, n2, acc);
        }
        if constexpr (HIST) {
          // vectors whose maximum reaches the window's floor are listed, then counted 32 at a time
          const float fv = __uint_as_float((t2 & 0xFFFFu) << 16);
          uint32_t cm = 0u;
#pragma unroll
          for (int u = 0; u < kSUnroll; ++u) {
            const uint32_t m2 = bmax2_nan(bmax2_nan(q[u].x, q[u].y), bmax2_nan(q[u].z, q[u].w));
            const float vm = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
            const int v = base + u * kThreads + tid;
            cm |= (vm >= fv && v < v_hi) ? (1u << u) : 0u;
          }
          if (__any_sync(kFullMask, cm != 0u)) {  // (the list holds fewer than 32 before: room for 32 per vector slot)
#pragma unroll
            for (int u = 0; u < kSUnroll; ++u) {
              const bool mine = (cm >> u) & 1u;
              const unsigned bal = __ballot_sync(kFullMask, mine);
              if (mine) {
                const int o = nl + __popc(bal & ((1u << lane) - 1u));
                wl[o] = q[u];
                wi[o] = base + u * kThreads + tid;
              }
              nl += __popc(bal);
            }
          }
        }
        float s0, s1;
        upk2(acc, s0, s1);
        z = df_add(z, s0 + s1);
        if constexpr (HIST) {
          if (nl >= 32) {  // count the listed vectors (the loaded ones are no longer live here)
            __syncwarp();
            count_list(wl, wi, nl, wh, x, __uint_as_float((t2 & 0xFFFFu) << 16));
            nl = 0;
          }
        }
      } else {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int u = 0; u < kSUnroll; ++u) {
          s0 += mass(__uint_as_float(q[u].x), c, nmc) + mass(__uint_as_float(q[u].y), c, nmc);
          s1 += mass(__uint_as_float(q[u].z), c, nmc) + mass(__uint_as_float(q[u].w), c, nmc);
        }
        z = df_add(z, s0 + s1);
      }
    }

    if constexpr (HIST) {
      if (nl > 0) {
        __syncwarp();
        count_list(wl, wi, nl, wh, x, __uint_as_float((t2 & 0xFFFFu) << 16));
        nl = 0;
      }
    }
    // ---- the piece's record: maximum, mass, counts below its maximum key
    if (lane == 0) {
      s_m[warp] = Mw;
      s_nan[warp] = nanw;
      s_top[warp] = Pw;
      s_floor[warp] = Fw;
    }
    __syncthreads();
    float M = -INFINITY;
    uint32_t nn = 0u;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      M = fmaxf(M, s_m[w]);
      nn |= s_nan[w];
    }
    DF zs = (!nn && Mw > -INFINITY) ? df_mulf(z, ex2_approx((Mw - M) * c)) : df_make(0.f);
    zs = warp_sum_df(zs);
    if (lane == 0) s_z[warp] = zs;
    __syncthreads();
    PieceRec* const rec = piece_rec(a, static_cast<int>(blockIdx.x), row);
    const uint32_t P = (HIST && M > -INFINITY) ? bkey(__float_as_uint(M) >> 16) : 0u;
    if (tid == 0) {
      DF zt = df_make(0.f);
#pragma unroll
      for (int w = 0; w < kWarps; ++w) zt = df_add(zt, s_z[w]);
      zt = df_norm(zt);
      rec->m = M;
      rec->zh = zt.hi;
      rec->zl = zt.lo;
      rec->top = P;
      rec->nan = nn;
    }
    if constexpr (HIST) {
      const bool has_x = x >= v_lo * PV && x < v_hi * PV;
      uint32_t* const bh = before_hist(a, row);
      for (int j = tid; j < kSW; j += kThreads) {
        uint32_t tot = 0u, bef = 0u;
        if (!nn && M > -INFINITY && P >= static_cast<uint32_t>(j)) {
          const uint32_t key = P - static_cast<uint32_t>(j);
#pragma unroll
          for (int w = 0; w < kWarps; ++w) {
            if (s_m[w] > -INFINITY && key >= s_floor[w] && key <= s_top[w]) {
              const uint32_t sl = key & static_cast<uint32_t>(kSW - 1);
              const uint32_t* const hw = hist + w * kSW;
              const uint32_t sh16 = 16u * (sl & 1u);
              const uint32_t a0 = (hw[sl >> 1] >> sh16) & 0xFFFFu, b0 = (hw[kSW / 2 + (sl >> 1)] >> sh16) & 0xFFFFu;
              bef += a0;
              tot += a0 + b0;
            }
          }
        }
        rec->hist[j] = tot;
        if (has_x) bh[j] = bef;
      }
    }
    __syncthreads();  // (the windows and the per-warp values are reused by the next piece)
  }
}

// ------------------------------------------------------------ row kernel

struct RowShmS {
  float pm[kMaxPiecesPerRow];
  uint32_t ptop[kMaxPiecesPerRow];
  float pzh[kMaxPiecesPerRow], pzl[kMaxPiecesPerRow];
  uint32_t pnan[kMaxPiecesPerRow];
  uint32_t wu[kWarps][2];
  DF wd[kWarps][2];
  float M;
  DF Z;
  int bad;
  uint32_t P;
  // a cut: found, its key, tokens of it kept, tokens of it in the row (or
  // in the set), the mass of the kept set, the draft token's rank in it
  int found;
  uint32_t kstar;
  int keep, gcount;
  DF zkept;
  int jbin;
  uint32_t rank_x;
  int rank_known;
  // below-window search: exact counts of one window of keys
  uint32_t fh[2][kSW];
};

// Exclusive scan of one count per thread (thread order) and the CTA total.
__device__ __forceinline__ uint32_t cta_excl_u(RowShmS& sh, uint32_t v, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = warp_incl_scan_u(v);
  if (lane == 31) sh.wu[warp][0] = incl;
  __syncthreads();
  uint32_t off = 0u, tot = 0u;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t t = sh.wu[w][0];
    if (w < warp) off += t;
    tot += t;
  }
  __syncthreads();
  total = tot;
  return off + incl - v;
}
// The same for a double-float per thread.
__device__ __forceinline__ DF cta_excl_df(RowShmS& sh, DF v, DF& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const DF incl = warp_incl_scan_df(v);
  if (lane == 31) sh.wd[warp][0] = incl;
  __syncthreads();
  DF off = df_make(0.f), tot = df_make(0.f);
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const DF t = sh.wd[w][0];
    if (w < warp) off = df_add(off, t);
    tot = df_add(tot, t);
  }
  __syncthreads();
  total = df_norm(tot);
  return df_norm(df_add(df_add(off, incl), df_neg(v)));
}
__device__ __forceinline__ DF cta_sum_df(RowShmS& sh, DF v) {
  DF t;
  (void)cta_excl_df(sh, v, t);
  return t;
}
__device__ __forceinline__ uint32_t cta_sum_u(RowShmS& sh, uint32_t v) {
  uint32_t t;
  (void)cta_excl_u(sh, v, t);
  return t;
}

// Tokens of a group kept by a mass target: the c-th token (0-based) has mass
// before + c e before it and is kept iff that is below the target.
__device__ __forceinline__ int keep_of(DF target, DF before, float e, int n) {
  const float need = df_f(df_norm(df_add(target, df_neg(before)))) / e;
  int kept = need >= static_cast<float>(n) ? n : static_cast<int>(ceilf(need));
  return max(1, min(kept, n));
}

// The cut below the window (keys < F), searched in the row itself: windows
// of kSW keys from just below F downwards, each one pass over the row with
// exact counts of its keys (kept apart before and from the draft token) and
// the largest key below it, where the next window starts.  The running totals
// start at cnt_above / mass_above (everything at or above F) and grow by each
// window's counts times its values' masses.  kind 0: count target ktarget
// (top-k); kind 1: mass target mtarget (top-p).  With lim_key != 0 only keys
// from lim_key up count, and of key lim_key only the first lim_keep tokens.
// Result in sh.found (1: cut found; 2: the whole set is kept) / kstar / keep /
// gcount / zkept / rank_x.
template <int DT>
__device__ void search_below(const SampleArgs& a, RowShmS& sh, const RowRef& rr, float c, float nmc, uint32_t F,
                             int kind, uint32_t cnt_above, DF mass_above, uint32_t ktarget, DF mtarget,
                             uint32_t lim_key, int lim_keep) {
  using E = Elt<DT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nv = a.V / E::kPerVec;
  const uint4* const vp = reinterpret_cast<const uint4*>(rr.ptr);
  const int x = rr.x;
  uint32_t cc = cnt_above;
  DF mc = mass_above;
  bool more = F > lim_key && F > 0u;
  uint32_t top = more ? F - 1u : 0u;
  if (tid == 0) sh.found = 0;
  __syncthreads();
  for (int pass = 0; pass < 160 && more; ++pass) {
    const uint32_t lo = max(top >= static_cast<uint32_t>(kSW - 1) ? top - static_cast<uint32_t>(kSW - 1) : 0u, lim_key);
    for (int j = tid; j < 2 * kSW; j += kThreads) (&sh.fh[0][0])[j] = 0u;
    __syncthreads();
    uint32_t below = 0u;  // largest key under the window (+1; 0: none)
    for (int v0 = tid; v0 < nv; v0 += kThreads * 8) {
      uint4 q8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + u * kThreads;
        q8[u] = v < nv ? ldg_stream(vp + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + u * kThreads;
        if (v >= nv) break;
#pragma unroll
        for (int j = 0; j < E::kPerVec; ++j) {
          const uint32_t key = E::key(E::bits_of(q8[u], j));
          if (key >= lo && key <= top)
            red_add_shared(smem_addr(&sh.fh[(v * E::kPerVec + j) >= x ? 1 : 0][top - key]), 1u);
          else if (key < lo)
            below = max(below, key + 1u);
        }
      }
    }
    below = __reduce_max_sync(kFullMask, below);
    if (lane == 0) sh.wu[warp][1] = below;
    __syncthreads();
    // the window's groups from the top: thread t holds keys top - 2t, top - 2t - 1
    uint32_t n2[2];
    float e2[2];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = 2 * tid + jj;
      const uint32_t key = top - static_cast<uint32_t>(j);
      n2[jj] = 0u;
      e2[jj] = 0.f;
      if (top >= static_cast<uint32_t>(j) && key >= lo) {
        n2[jj] = sh.fh[0][j] + sh.fh[1][j];
        if (lim_key != 0u && key == lim_key) n2[jj] = min(n2[jj], static_cast<uint32_t>(lim_keep));
        e2[jj] = mass(bval_of_key(key), c, nmc);
      }
    }
    uint32_t ntot;
    const uint32_t cex = cc + cta_excl_u(sh, n2[0] + n2[1], ntot);
    const DF m0 = df_make(static_cast<float>(n2[0]) * e2[0]);
    const DF mine = df_add(m0, static_cast<float>(n2[1]) * e2[1]);
    DF mtot;
    const DF mex = df_norm(df_add(mc, cta_excl_df(sh, mine, mtot)));
    // the group where the running total reaches the target (one thread at most)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const uint32_t cb = jj == 0 ? cex : cex + n2[0];
      const DF mb = jj == 0 ? mex : df_norm(df_add(mex, m0));
      if (n2[jj] == 0u) continue;
      const uint32_t ca = cb + n2[jj];
      const DF ma = df_norm(df_add(mb, static_cast<float>(n2[jj]) * e2[jj]));
      const bool hit = kind == 0 ? (cb < ktarget && ca >= ktarget) : (df_lt(mb, mtarget) && !df_lt(ma, mtarget));
      if (hit) {
        const int kept = kind == 0 ? static_cast<int>(ktarget - cb) : keep_of(mtarget, mb, e2[jj], static_cast<int>(n2[jj]));
        const int j = 2 * tid + jj;
        sh.found = 1;
        sh.kstar = top - static_cast<uint32_t>(j);
        sh.keep = kept;
        sh.gcount = static_cast<int>(n2[jj]);
        sh.zkept = df_norm(df_add(mb, static_cast<float>(kept) * e2[jj]));
        sh.rank_x = sh.fh[0][j];
        sh.rank_known = 1;
      }
    }
    __syncthreads();
    if (sh.found) break;
    cc += ntot;
    mc = df_norm(df_add(mc, mtot));
    uint32_t nb = 0u;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) nb = max(nb, sh.wu[w][1]);
    more = nb > 0u && nb - 1u >= lim_key && lo > lim_key;
    top = nb - 1u;
    __syncthreads();
  }
  if (tid == 0 && !sh.found) {  // nothing left below (the rounding of a total): the whole set is kept
    sh.found = 2;
    sh.zkept = mc;
  }
  __syncthreads();
}

// One CTA per row: merge the row's piece records, decide the kept set, p(x).
template <int DT, bool HIST>
__global__ void __launch_bounds__(kThreads, 4) split_row_kernel(const SampleArgs a) {
  using E = Elt<DT>;
  constexpr int PV = E::kPerVec;
  __shared__ RowShmS sh;
  const int tid = threadIdx.x;
  const int row = static_cast<int>(blockIdx.x);
  const RowRef rr = row_ref(a, row, E::kBytes);
  const float c = row_c(a, rr.b);
  const int R = a.B * (2 * a.k + 1);
  const long long nvr = a.V / PV;
  const long long units = static_cast<long long>(R) * nvr;
  const int grid = a.split_grid;
  const int first = cta_of(units, grid, static_cast<long long>(row) * nvr);
  const int last = cta_of(units, grid, static_cast<long long>(row + 1) * nvr - 1);
  const int np = min(last - first + 1, kMaxPiecesPerRow);
  // the draft token's value, read early (thread 0 publishes p(x))
  const uint32_t xb = (tid == 0 && rr.x >= 0) ? E::bits_at(rr.ptr, rr.x) : 0u;
  if (tid < np) {
    const PieceRec* r = piece_rec(a, first + tid, row);
    sh.pm[tid] = __ldcg(&r->m);
    sh.pzh[tid] = __ldcg(&r->zh);
    sh.pzl[tid] = __ldcg(&r->zl);
    sh.ptop[tid] = __ldcg(&r->top);
    sh.pnan[tid] = __ldcg(&r->nan);
  }
  __syncthreads();
  if (tid == 0) {
    float M = -INFINITY;
    uint32_t nn = 0u;
    for (int p = 0; p < np; ++p) {
      M = fmaxf(M, sh.pm[p]);
      nn |= sh.pnan[p];
    }
    DF Z = df_make(0.f);
    if (M > -INFINITY)
      for (int p = 0; p < np; ++p)
        if (sh.pm[p] > -INFINITY) Z = df_add(Z, df_mulf(DF{sh.pzh[p], sh.pzl[p]}, ex2_approx((sh.pm[p] - M) * c)));
    sh.M = M;
    sh.Z = df_norm(Z);
    sh.bad = (nn != 0u || !(M > -INFINITY) || !(M < INFINITY) || !(c > 0.f)) ? 1 : 0;
    sh.P = (HIST && M > -INFINITY && M < INFINITY) ? bkey(__float_as_uint(M) >> 16) : 0u;
    sh.found = 0;
    sh.rank_known = 0;
    sh.rank_x = 0u;
  }
  __syncthreads();
  const float M = sh.M;
  const float nmc = -M * c;
  const bool bad = sh.bad != 0;
  const bool filt = HIST && (a.top_k > 0 || a.top_p < 1.f);
  // the kept set, decided below (thread 0's copy is the one published)
  int all_kept = 1;
  uint32_t kstar = 0u;
  int keep = 0, gcount = 0;
  DF zkept = sh.Z;

  if (filt && !bad) {
    const uint32_t P = sh.P;
    // every piece counted its keys down to F at least (its own floor is not above the row's)
    const uint32_t F = band_floor(M, P, c);
    // the row's window counts: thread t holds keys P - 2t and P - 2t - 1
    uint32_t cnt[2];
    float e[2];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = 2 * tid + jj;
      cnt[jj] = 0u;
      e[jj] = 0.f;
      if (P >= static_cast<uint32_t>(j) && P - static_cast<uint32_t>(j) >= F) {
        for (int p = 0; p < np; ++p) {
          const uint32_t d = P - sh.ptop[p];
          if (sh.pm[p] > -INFINITY && static_cast<uint32_t>(j) >= d)
            cnt[jj] += __ldcg(&piece_rec(a, first + p, row)->hist[j - static_cast<int>(d)]);
        }
        e[jj] = mass(bval_of_key(P - static_cast<uint32_t>(j)), c, nmc);
      }
    }
    uint32_t setc[2] = {cnt[0], cnt[1]};
    // ---- top-k: the group where the count from the top reaches top_k
    bool k_on = a.top_k > 0, k_in = false, k_below = false;
    uint32_t kk = 0u, rank_k = 0u;
    int keep_k = 0, gk = 0;
    DF Zk = sh.Z;
    if (k_on) {
      uint32_t wtot;
      const uint32_t excl = cta_excl_u(sh, cnt[0] + cnt[1], wtot);
      const uint32_t K = static_cast<uint32_t>(a.top_k);
      if (excl < K && excl + cnt[0] + cnt[1] >= K) {
        const int jj = excl + cnt[0] >= K ? 0 : 1;
        sh.found = 1;
        sh.jbin = 2 * tid + jj;
        sh.keep = static_cast<int>(K - (jj == 0 ? excl : excl + cnt[0]));
        sh.gcount = static_cast<int>(cnt[jj]);
      }
      __syncthreads();
      if (sh.found) {
        k_in = true;
        const int jk = sh.jbin;
        kk = P - static_cast<uint32_t>(jk);
        keep_k = sh.keep;
        gk = sh.gcount;
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int j = 2 * tid + jj;
          setc[jj] = j < jk ? cnt[jj] : (j == jk ? static_cast<uint32_t>(keep_k) : 0u);
        }
        const DF mine = df_add(df_make(static_cast<float>(setc[0]) * e[0]), static_cast<float>(setc[1]) * e[1]);
        Zk = cta_sum_df(sh, mine);
      } else {
        // below the window: the whole window is in the top-k set
        const DF mine = df_add(df_make(static_cast<float>(cnt[0]) * e[0]), static_cast<float>(cnt[1]) * e[1]);
        const DF wm = cta_sum_df(sh, mine);
        search_below<DT>(a, sh, rr, c, nmc, F, 0, wtot, wm, K, df_make(0.f), 0u, 0);
        k_below = true;
        kk = sh.kstar;
        keep_k = sh.keep;
        gk = sh.gcount;
        Zk = sh.zkept;
        rank_k = sh.rank_x;
        if (sh.found == 2) {  // (not reached: the count target is exact)
          k_on = false;
          k_below = false;
          Zk = sh.Z;
        }
      }
      __syncthreads();
      if (tid == 0) {
        sh.found = 0;
        sh.rank_known = 0;  // (the rank at the final cut is taken below)
      }
      __syncthreads();
    }
    // ---- top-p over the top-k set: the group where the mass reaches top_p Zk
    if (a.top_p < 1.f) {
      const DF target = df_mulf(Zk, a.top_p);
      const DF m0 = df_make(static_cast<float>(setc[0]) * e[0]);
      const DF mine = df_add(m0, static_cast<float>(setc[1]) * e[1]);
      DF wm;
      const DF before = cta_excl_df(sh, mine, wm);
      const DF incl0 = df_norm(df_add(before, m0));
      const DF incl1 = df_norm(df_add(before, mine));
      if (df_lt(before, target) && !df_lt(incl1, target)) {
        const int jj = !df_lt(incl0, target) ? 0 : 1;
        const DF bj = jj == 0 ? before : incl0;
        sh.found = 1;
        sh.jbin = 2 * tid + jj;
        sh.keep = keep_of(target, bj, e[jj], static_cast<int>(setc[jj]));
        sh.gcount = static_cast<int>(cnt[jj]);
        sh.zkept = df_norm(df_add(bj, static_cast<float>(sh.keep) * e[jj]));
      }
      __syncthreads();
      if (sh.found) {
        all_kept = 0;
        kstar = P - static_cast<uint32_t>(sh.jbin);
        keep = sh.keep;
        gcount = sh.gcount;
        zkept = sh.zkept;
      } else if (k_in) {  // (rounding) the whole top-k set
        all_kept = 0;
        kstar = kk;
        keep = keep_k;
        gcount = gk;
        zkept = Zk;
      } else {
        uint32_t wc = cta_sum_u(sh, setc[0] + setc[1]);
        search_below<DT>(a, sh, rr, c, nmc, F, 1, wc, wm, 0u, target, k_on ? kk : 0u, k_on ? keep_k : 0);
        if (sh.found == 1) {
          all_kept = 0;
          kstar = sh.kstar;
          keep = sh.keep;
          gcount = sh.gcount;
          zkept = sh.zkept;
        } else if (k_on) {  // (rounding) the whole top-k set
          all_kept = 0;
          kstar = kk;
          keep = keep_k;
          gcount = gk;
          zkept = Zk;
          if (tid == 0) {
            sh.rank_x = rank_k;
            sh.rank_known = 1;
          }
        } else {
          all_kept = 1;
          zkept = sh.Z;
        }
      }
    } else if (k_on) {
      all_kept = 0;
      kstar = kk;
      keep = keep_k;
      gcount = gk;
      zkept = Zk;
      if (k_below && tid == 0) {
        sh.rank_x = rank_k;
        sh.rank_known = 1;
      }
    }
    // the draft token's rank in the cut group, from the counts before it
    if (!all_kept && !sh.rank_known && rr.x >= 0 && tid == 0) {
      uint32_t rank = 0u;
      for (int p = 0; p < np; ++p) {
        const int cta = first + p;
        const long long rb = static_cast<long long>(row) * nvr;
        const long long s0 = max(range_start(units, grid, cta), rb) - rb;
        const long long s1 = min(range_start(units, grid, cta + 1), rb + nvr) - rb;
        if (!(sh.pm[p] > -INFINITY) || sh.ptop[p] < kstar || sh.ptop[p] - kstar >= static_cast<uint32_t>(kSW)) continue;
        const int d = static_cast<int>(sh.ptop[p] - kstar);
        if (s1 * PV <= rr.x) rank += __ldcg(&piece_rec(a, cta, row)->hist[d]);
        else if (s0 * PV <= rr.x) rank += __ldcg(before_hist(a, row) + d);
      }
      sh.rank_x = rank;
    }
  }
  __syncthreads();

  // ---- publish: the kept set and the probability at the draft token
  if (tid == 0) {
    SRow o = {};
    o.m = M;
    o.c = c;
    o.bad = bad ? 1 : 0;
    o.all_kept = all_kept;
    o.kstar = kstar;
    o.keep = keep;
    o.gcount = gcount;
    o.zkh = zkept.hi;
    o.zkl = zkept.lo;
    const float zk = df_f(zkept);
    o.izk = (!bad && zk > 0.f) ? 1.f / zk : 0.f;
    float xp = 0.f;
    if (!bad && rr.x >= 0) {
      const uint32_t kx = E::key(xb);
      const bool kept = all_kept || kx > kstar || (kx == kstar && sh.rank_x < static_cast<uint32_t>(keep));
      if (kept) xp = mass(E::value(xb), c, nmc) / zk;
    }
    o.xprob = xp;
    *reinterpret_cast<SRow*>(a.hdrs + row) = o;
    if (rr.i < a.k) {
      if (rr.target && a.out_p) a.out_p[static_cast<size_t>(rr.b) * a.k + rr.i] = xp;
      if (!rr.target && a.out_q) a.out_q[static_cast<size_t>(rr.b) * a.k + rr.i] = xp;
    }
    uint32_t st = bad ? SPEC_STATUS_BAD_ROW : 0u;
    if (rr.target && rr.i < a.k && rr.x < 0) st |= SPEC_STATUS_BAD_TOKEN;
    if (st) set_status(a.status, st);
  }
  // ---- leave the records read here zeroed
  if (HIST) {
    for (int p = 0; p < np; ++p) {
      uint32_t* h = piece_rec(a, first + p, row)->hist;
      for (int j = tid; j < kSW; j += kThreads) h[j] = 0u;
    }
    if (rr.x >= 0)
      for (int j = tid; j < kSW; j += kThreads) before_hist(a, row)[j] = 0u;
  }
  if (tid < np) {
    PieceRec* r = piece_rec(a, first + tid, row);
    r->m = 0.f;
    r->zh = 0.f;
    r->zl = 0.f;
    r->top = 0u;
    r->nan = 0u;
  }
}

// ------------------------------------------------------------ draw kernel

struct DrawShm {
  uint64_t bar;            // the slices' bulk copies
  uint32_t ties[2];        // this CTA's tokens of the two cut keys (read by the cluster)
  float sum_hi, sum_lo;    // this CTA's residual mass (read by the cluster)
  uint32_t wt[kDrawWarps][2];  // per warp: tokens of the cut keys
  DF ws[kDrawWarps];           // per warp: residual mass
  float pick_hi, pick_lo;  // residual mass before the picked warp
  float all_hi[kDrawCl], all_lo[kDrawCl];  // every CTA's residual mass
  // per warp: vectors that hold a token of P's kept set, in index order, with
  // the ranks of their first cut-key tokens (slice vector, rank in P, rank in Q)
  uint32_t lv[kDrawWarps][64];
  uint32_t lr[kDrawWarps][64][2];
  uint32_t cta_ties[2];    // cut-key tokens before this CTA
  int n;
  int pick_warp;
  int token;
};

// The kept test of one token: key above the cut, or of the cut key with a
// rank below the tokens kept.
__device__ __forceinline__ bool kept_tok(const SRow& r, uint32_t key, uint32_t rank) {
  return r.all_kept || key > r.kstar || (key == r.kstar && rank < static_cast<uint32_t>(r.keep));
}

// max(0, p - q) of one token from its two masses and the rows' inverse kept
// masses, rounded step by step (no contraction): the sums over the cluster and
// the walk to the token use this one function, so they agree bit for bit.
__device__ __forceinline__ float resid_weight(float mp, float izp, float mq, float izq) {
  return fmaxf(__fsub_rn(__fmul_rn(mp, izp), __fmul_rn(mq, izq)), 0.f);
}

// Residual weights of the tokens of one vector pair, in index order; rp / rq:
// ranks of this vector's first cut-key token in each row.
template <int DT>
__device__ __forceinline__ void pair_weights(const uint4& vp_, const uint4& vq_, const SRow& P, const SRow& Q,
                                             bool use_q, uint32_t rp, uint32_t rq, float* w) {
  using E = Elt<DT>;
  const float nmp = -P.m * P.c, nmq = use_q ? -Q.m * Q.c : 0.f;
#pragma unroll
  for (int j = 0; j < E::kPerVec; ++j) {
    const uint32_t bp = E::bits_of(vp_, j);
    const uint32_t kp = E::key(bp);
    const bool kpk = kept_tok(P, kp, rp);
    rp += (kp == P.kstar) ? 1u : 0u;
    const float mp = kpk ? mass(E::value(bp), P.c, nmp) : 0.f;
    float mq = 0.f;
    if (use_q) {
      const uint32_t bq = E::bits_of(vq_, j);
      const uint32_t kq = E::key(bq);
      const bool kqk = kept_tok(Q, kq, rq);
      rq += (kq == Q.kstar) ? 1u : 0u;
      mq = kqk ? mass(E::value(bq), Q.c, nmq) : 0.f;
    }
    w[j] = kpk ? resid_weight(mp, P.izk, mq, Q.izk) : 0.f;
  }
}
// Sum of the residual weights of one vector pair (the same values as
// pair_weights, added in index order): P's kept tokens are found by value
// first, and only they are weighed.
template <int DT>
__device__ __forceinline__ float pair_sum(const uint4& vp_, const uint4& vq_, const SRow& P, const SRow& Q, bool use_q,
                                          uint32_t rp, uint32_t rq) {
  using E = Elt<DT>;
  uint32_t kmask = 0u, qmask = 0u;  // P's kept tokens; Q's kept tokens
#pragma unroll
  for (int j = 0; j < E::kPerVec; ++j) {
    const uint32_t kp = E::key(E::bits_of(vp_, j));
    kmask |= kept_tok(P, kp, rp) ? (1u << j) : 0u;
    rp += (kp == P.kstar) ? 1u : 0u;
    if (use_q) {
      const uint32_t kq = E::key(E::bits_of(vq_, j));
      qmask |= kept_tok(Q, kq, rq) ? (1u << j) : 0u;
      rq += (kq == Q.kstar) ? 1u : 0u;
    }
  }
  const float nmp = -P.m * P.c, nmq = use_q ? -Q.m * Q.c : 0.f;
  float sum = 0.f;
  while (kmask) {
    const int j = __ffs(kmask) - 1;
    kmask &= kmask - 1u;
    const float mp = mass(E::value(E::bits_of(vp_, j)), P.c, nmp);
    const float mq = ((qmask >> j) & 1u) ? mass(E::value(E::bits_of(vq_, j)), Q.c, nmq) : 0.f;
    sum += resid_weight(mp, P.izk, mq, Q.izk);
  }
  return sum;
}

template <int DT>
__device__ __forceinline__ uint32_t ties_of(const uint4& v, uint32_t kstar) {
  using E = Elt<DT>;
  if constexpr (DT == DT_BF16) {
    // tokens whose value equals the cut value: equal 16-bit patterns, and
    // for the value 0 both signed zeros
    const uint32_t kb = E::bits_of_key(kstar);
    const uint32_t k2 = kb | (kb << 16);
    const bool zero = (kb & 0x7FFFu) == 0u;
    uint32_t n = 0u;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t wd = word_of(v, w);
      uint32_t eq = __vcmpeq2(wd, k2);
      if (zero) eq |= __vcmpeq2(wd, 0u) | __vcmpeq2(wd, 0x80008000u);
      n += __popc(eq);
    }
    return n >> 4;
  } else {
    uint32_t n = 0u;
#pragma unroll
    for (int j = 0; j < E::kPerVec; ++j) n += E::key(E::bits_of(v, j)) == kstar ? 1u : 0u;
    return n;
  }
}

// Exclusive ranks of this lane's cut-key tokens within one round of 32
// vectors (one per lane), both rows packed 16 + 16 bits, and the round's
// totals: a ballot when no lane holds more than one, else a scan.
__device__ __forceinline__ void round_ranks(uint32_t lp, uint32_t lq, uint32_t& ep, uint32_t& eq, uint32_t& tp,
                                            uint32_t& tq) {
  const int lane = threadIdx.x & 31;
  if (__any_sync(kFullMask, lp > 1u || lq > 1u)) {
    const uint32_t both = lp | (lq << 16);
    const uint32_t incl = warp_incl_scan_u(both);
    const uint32_t ex = incl - both, tot = __shfl_sync(kFullMask, incl, 31);
    ep = ex & 0xFFFFu;
    eq = ex >> 16;
    tp = tot & 0xFFFFu;
    tq = tot >> 16;
  } else {
    const unsigned bp = __ballot_sync(kFullMask, lp != 0u), bq = __ballot_sync(kFullMask, lq != 0u);
    const unsigned lt = (1u << lane) - 1u;
    ep = __popc(bp & lt);
    eq = __popc(bq & lt);
    tp = __popc(bp);
    tq = __popc(bq);
  }
}

// Largest value of a 16-byte vector (NaN-propagating).
template <int DT>
__device__ __forceinline__ float vec_max(const uint4& v) {
  if constexpr (DT == DT_BF16) {
    const uint32_t m2 = bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w));
    return max_nan(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
  } else {
    return max_nan(max_nan(__uint_as_float(v.x), __uint_as_float(v.y)), max_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
}

// Walks a warp's segment [s0, s1) of the slice in rounds of 32 vectors,
// keeping the ranks of the two cut keys' tokens in index order, and lists the
// vectors that can hold a token of P's kept set (maximum at or above pcut);
// every 32 listed vectors (and the rest at the end) go to f(n, v, rp, rq) as
// one batch, lane l holding the l-th (v: slice vector; rp, rq: ranks of its
// first cut-key tokens) if l < n.  f returns true to stop.  The weights of the
// other vectors are 0, so only the listed ones are evaluated.
template <int DT, typename F>
__device__ __forceinline__ void walk_listed(uint32_t* lv, uint32_t (*lr)[2], uint32_t sp, uint32_t sq, int s0, int s1,
                                            bool pt, bool qt, const SRow& P, const SRow& Q, bool use_q, float pcut,
                                            uint32_t rp, uint32_t rq, F&& f) {
  const int lane = threadIdx.x & 31;
  int cnt = 0;
  bool stop = false;
  for (int v0 = s0; v0 < s1 && !stop; v0 += 32) {
    const int v = v0 + lane;
    uint32_t lp = 0u, lq = 0u;
    bool keep = false;
    if (v < s1) {
      const uint4 xp = lds128(sp + 16u * v);
      if (pt) lp = ties_of<DT>(xp, P.kstar);
      if (use_q && qt) lq = ties_of<DT>(lds128(sq + 16u * v), Q.kstar);
      keep = vec_max<DT>(xp) >= pcut;
    }
    uint32_t ep = 0u, eq = 0u, tp = 0u, tq = 0u;
    if (pt || qt) round_ranks(lp, lq, ep, eq, tp, tq);
    const unsigned bal = __ballot_sync(kFullMask, keep);
    if (keep) {
      const int o = cnt + __popc(bal & ((1u << lane) - 1u));
      lv[o] = static_cast<uint32_t>(v);
      lr[o][0] = rp + ep;
      lr[o][1] = rq + eq;
    }
    cnt += __popc(bal);
    rp += tp;
    rq += tq;
    __syncwarp();
    if (cnt >= 32) {
      const bool in = true;
      stop = f(32, in ? lv[lane] : 0u, lr[lane][0], lr[lane][1]);
      __syncwarp();
      cnt -= 32;
      if (lane < cnt) {  // (at most 31 left: move them to the front)
        const uint32_t a0 = lv[32 + lane], a1 = lr[32 + lane][0], a2 = lr[32 + lane][1];
        __syncwarp(__activemask());
        lv[lane] = a0;
        lr[lane][0] = a1;
        lr[lane][1] = a2;
      }
      __syncwarp();
    }
  }
  if (!stop && cnt > 0) {
    const uint32_t a0 = lane < cnt ? lv[lane] : 0u, a1 = lane < cnt ? lr[lane][0] : 0u, a2 = lane < cnt ? lr[lane][1] : 0u;
    f(cnt, a0, a1, a2);
  }
  __syncwarp();
}

// Vectors of a CTA's slice (the largest slice of the cluster).
__host__ __device__ __forceinline__ int draw_slice_vecs(int nv) { return (nv + kDrawCl - 1) / kDrawCl; }

// One cluster of kDrawCl CTAs per sequence: the first rejection n, the
// committed tokens, and the draw at n (see the file comment).  Each CTA
// bulk-copies its slice of the row pair into shared memory once; every
// later step reads it there.
template <int DT>
__global__ void __launch_bounds__(kDrawThreads) split_draw_kernel(const SampleArgs a) {
  using E = Elt<DT>;
  constexpr int PV = E::kPerVec;
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ DrawShm sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = static_cast<int>(blockIdx.x) / kDrawCl;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k, V = a.V;
  const int rt0 = b * (k + 1), rd0 = a.B * (k + 1) + b * k;
  const int32_t* const x = a.tokens + static_cast<size_t>(b) * k;

  // ---- n: the first position whose test fails (k <= 31: one warp)
  if (warp == 0) {
    bool rej = false;
    if (lane < k) {
      const SRow* rp = reinterpret_cast<const SRow*>(a.hdrs + rt0 + lane);
      const SRow* rq = reinterpret_cast<const SRow*>(a.hdrs + rd0 + lane);
      const float px = rp->xprob, qx = rq->xprob;
      const int bp = rp->bad, bq = rq->bad;
      const float u = a.uniforms[static_cast<size_t>(b) * (k + 2) + lane];
      const bool xok = x[lane] >= 0 && x[lane] < V;
      rej = !(!bp && !bq && xok && u * qx < px);
    }
    const unsigned rb = __ballot_sync(kFullMask, rej);
    if (lane == 0) sh.n = rb ? __ffs(rb) - 1 : k;
  }
  if (tid == 0) {
    mbar_init(&sh.bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int n = sh.n;
  const bool use_q = n < k;
  // (written by the previous launch)
  const SRow P = *reinterpret_cast<const SRow*>(a.hdrs + rt0 + n);
  const SRow Q = use_q ? *reinterpret_cast<const SRow*>(a.hdrs + rd0 + n) : P;
  const bool bad = P.bad || (use_q && Q.bad);
  const float u = a.uniforms[static_cast<size_t>(b) * (k + 2) + (use_q ? k + 1 : k)];
  const size_t rbytes = static_cast<size_t>(V) * E::kBytes;
  const unsigned char* const gp = static_cast<const unsigned char*>(a.target) + static_cast<size_t>(rt0 + n) * rbytes;
  const unsigned char* const gq =
      use_q ? static_cast<const unsigned char*>(a.draft) + static_cast<size_t>(b * k + n) * rbytes : gp;
  // this CTA's slice (row vectors [c0, c1)) in shared memory: P, then Q
  const int nv = V / PV;
  const int c0 = static_cast<int>(static_cast<long long>(rank) * nv / kDrawCl);
  const int c1 = static_cast<int>(static_cast<long long>(rank + 1) * nv / kDrawCl);
  const uint32_t sp = smem_addr(dsm), sq = sp + static_cast<uint32_t>(draw_slice_vecs(nv)) * 16u;
  const uint32_t bytes = static_cast<uint32_t>(c1 - c0) * 16u;
  const bool copy = !bad && bytes > 0u;
  if (copy && tid == 0) {
    mbar_arrive_expect_tx(&sh.bar, use_q ? 2u * bytes : bytes);
    bulk_copy_g2s_addr(sp, gp + static_cast<size_t>(c0) * 16u, bytes, &sh.bar);
    if (use_q) bulk_copy_g2s_addr(sq, gq + static_cast<size_t>(c0) * 16u, bytes, &sh.bar);
  }
  const bool landed = !copy || mbar_wait_bounded(&sh.bar, 0u);
  const bool lost = __syncthreads_or(!landed) != 0;  // a copy that never landed: this slice counts as empty
  if (lost && tid == 0) set_status(a.status, SPEC_STATUS_TIMEOUT);
  // this warp's contiguous segment of the slice (slice-relative vectors)
  const int len = lost ? 0 : c1 - c0;
  const int s0 = static_cast<int>(static_cast<long long>(warp) * len / kDrawWarps);
  const int s1 = static_cast<int>(static_cast<long long>(warp + 1) * len / kDrawWarps);
  const bool pt = !P.all_kept && P.keep < P.gcount;
  // a vector whose maximum lies under P's cut value holds no token of P's kept set: its weights are 0
  const float pcut = (DT == DT_BF16 && !P.all_kept) ? bval_of_key(P.kstar) : -INFINITY;
  const bool qt = use_q && !Q.all_kept && Q.keep < Q.gcount;
  const bool ties = !bad && (pt || qt);

  // ---- ranks of the cut groups: tokens of each cut key before this warp's segment
  uint32_t base_p = 0u, base_q = 0u;
  if (ties) {
    uint32_t tp = 0u, tq = 0u;
    for (int v = s0 + lane; v < s1; v += 32) {
      if (pt) tp += ties_of<DT>(lds128(sp + 16u * v), P.kstar);
      if (qt) tq += ties_of<DT>(lds128(sq + 16u * v), Q.kstar);
    }
    tp = __reduce_add_sync(kFullMask, tp);
    tq = __reduce_add_sync(kFullMask, tq);
    if (lane == 0) {
      sh.wt[warp][0] = tp;
      sh.wt[warp][1] = tq;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t cp = 0u, cq = 0u;
      for (int w = 0; w < kDrawWarps; ++w) {
        cp += sh.wt[w][0];
        cq += sh.wt[w][1];
      }
      sh.ties[0] = cp;
      sh.ties[1] = cq;
    }
  }
  cluster.sync();
  if (ties) {
    if (tid == 0) {  // the tokens before this CTA, read once from the cluster
      uint32_t cp = 0u, cq = 0u;
      for (int r = 0; r < rank; ++r) {
        cp += ld_cluster_u32(mapa_shared(smem_addr(&sh.ties[0]), static_cast<uint32_t>(r)));
        cq += ld_cluster_u32(mapa_shared(smem_addr(&sh.ties[1]), static_cast<uint32_t>(r)));
      }
      sh.cta_ties[0] = cp;
      sh.cta_ties[1] = cq;
    }
    __syncthreads();
    base_p = sh.cta_ties[0];
    base_q = sh.cta_ties[1];
    for (int w = 0; w < warp; ++w) {
      base_p += sh.wt[w][0];
      base_q += sh.wt[w][1];
    }
  }

  // ---- residual mass per warp segment, then over the cluster
  // (mode 1: max(0, p - q); mode 0: p alone -- the bonus, or a residual that summed to 0)
  DF total = df_make(0.f), before = df_make(0.f);
  int mode = use_q ? 1 : 0;
  for (int pass = 0; pass < 2; ++pass) {
    DF wsum = df_make(0.f);
    if (!bad) {
      walk_listed<DT>(sh.lv[warp], sh.lr[warp], sp, sq, s0, s1, pt, qt, P, Q, mode == 1, pcut, base_p, base_q,
                      [&](int nb, uint32_t v, uint32_t rpv, uint32_t rqv) {
                        if (lane < nb) {
                          const uint4 xp = lds128(sp + 16u * v);
                          const uint4 xq = mode == 1 ? lds128(sq + 16u * v) : xp;
                          wsum = df_add(wsum, pair_sum<DT>(xp, xq, P, Q, mode == 1, rpv, rqv));
                        }
                        return false;
                      });
    }
    wsum = warp_sum_df(wsum);
    if (lane == 0) sh.ws[warp] = wsum;
    __syncthreads();
    if (tid == 0) {
      DF t = df_make(0.f);
      for (int w = 0; w < kDrawWarps; ++w) t = df_add(t, sh.ws[w]);
      t = df_norm(t);
      sh.sum_hi = t.hi;
      sh.sum_lo = t.lo;
    }
    cluster.sync();
    if (tid < kDrawCl) {  // every CTA's mass, read once from the cluster
      sh.all_hi[tid] = ld_cluster_f32(mapa_shared(smem_addr(&sh.sum_hi), static_cast<uint32_t>(tid)));
      sh.all_lo[tid] = ld_cluster_f32(mapa_shared(smem_addr(&sh.sum_lo), static_cast<uint32_t>(tid)));
    }
    __syncthreads();
    total = df_make(0.f);
    before = df_make(0.f);
    for (int r = 0; r < kDrawCl; ++r) {
      const DF o{sh.all_hi[r], sh.all_lo[r]};
      if (r < rank) before = df_add(before, o);
      total = df_add(total, o);
    }
    total = df_norm(total);
    before = df_norm(before);
    // (every CTA decides alike: the same sums, added in the same order)
    if (mode == 0 || total.hi > 0.f || bad) break;
    cluster.sync();  // (sum_hi / sum_lo are rewritten by the second pass)
    mode = 0;        // a residual that sums to 0 (rounding): draw from p
  }

  // ---- the token: the CTA whose range holds u S, its warp, its lane, its element
  const DF tgt = df_mulf(total, u);
  const DF mysum{sh.sum_hi, sh.sum_lo};
  const DF after = df_norm(df_add(before, mysum));
  // the CTA: before <= tgt < after (the last CTA with mass takes a target past the end)
  bool mine = !bad && mysum.hi > 0.f && !df_lt(tgt, before) && df_lt(tgt, after);
  if (!bad && mysum.hi > 0.f && !df_lt(tgt, after)) {
    bool later = false;
    for (int r = rank + 1; r < kDrawCl; ++r) later = later || sh.all_hi[r] > 0.f;
    mine = !later;
  }
  if (tid == 0) {
    sh.token = -1;
    sh.pick_warp = -1;
  }
  __syncthreads();
  if (mine) {
    if (tid == 0) {
      DF cm = before;
      int pw = -1;
      for (int w = 0; w < kDrawWarps; ++w) {
        const DF nc = df_norm(df_add(cm, sh.ws[w]));
        if (sh.ws[w].hi > 0.f) pw = w;
        if (sh.ws[w].hi > 0.f && df_lt(tgt, nc)) break;
        cm = nc;
      }
      sh.pick_warp = pw;
      sh.pick_hi = cm.hi;
      sh.pick_lo = cm.lo;
    }
    __syncthreads();
    if (warp == sh.pick_warp) {
      DF cm{sh.pick_hi, sh.pick_lo};
      int token = -1, last_tok = -1;  // (last_tok: the last token with mass, for a target past the end)
      walk_listed<DT>(sh.lv[warp], sh.lr[warp], sp, sq, s0, s1, pt, qt, P, Q, mode == 1, pcut, base_p, base_q,
                      [&](int nb, uint32_t v, uint32_t rpv, uint32_t rqv) -> bool {
                        float w[PV];
#pragma unroll
                        for (int j = 0; j < PV; ++j) w[j] = 0.f;
                        if (lane < nb) {
                          const uint4 xp = lds128(sp + 16u * v);
                          const uint4 xq = mode == 1 ? lds128(sq + 16u * v) : xp;
                          pair_weights<DT>(xp, xq, P, Q, mode == 1, rpv, rqv, w);
                        }
                        float ls = 0.f;
#pragma unroll
                        for (int j = 0; j < PV; ++j) ls += w[j];
                        // lanes in index order: the first lane whose running total passes the target
                        const DF li = warp_incl_scan_df(df_make(ls));
                        const DF lend = df_norm(df_add(cm, li));
                        const unsigned hit = __ballot_sync(kFullMask, ls > 0.f && df_lt(tgt, lend));
                        const unsigned any = __ballot_sync(kFullMask, ls > 0.f);
                        if (any) {
                          const int ll = 31 - __clz(any);
                          int lj = -1;
                          for (int j = 0; j < PV; ++j)
                            if (w[j] > 0.f) lj = j;
                          lj = __shfl_sync(kFullMask, lj, ll);
                          const uint32_t vl = __shfl_sync(kFullMask, v, ll);
                          last_tok = (c0 + static_cast<int>(vl)) * PV + lj;
                        }
                        if (hit) {
                          const int pl = __ffs(hit) - 1;
                          if (lane == pl) {
                            DF cc = df_norm(df_add(lend, df_neg(df_make(ls))));  // before this lane
                            int jl = -1;
                            for (int j = 0; j < PV; ++j) {
                              if (w[j] <= 0.f) continue;
                              jl = j;
                              const DF nc = df_norm(df_add(cc, w[j]));
                              if (df_lt(tgt, nc)) break;
                              cc = nc;
                            }
                            token = (c0 + static_cast<int>(v)) * PV + jl;
                          }
                          token = __shfl_sync(kFullMask, token, pl);
                          return true;
                        }
                        cm = df_norm(df_add(cm, shfl_df(li, 31)));
                        return false;
                      });
      if (lane == 0) sh.token = token >= 0 ? token : last_tok;
    }
    __syncthreads();
    if (tid == 0) a.out_tokens[static_cast<size_t>(b) * (k + 1) + n] = sh.token;
  }
  if (rank == 0) {
    int32_t* out = a.out_tokens + static_cast<size_t>(b) * (k + 1);
    for (int i = tid; i <= k; i += kDrawThreads) {
      if (i < n) out[i] = x[i];
      else if (i > n) out[i] = -1;
    }
    if (bad && tid == 0) out[n] = -1;
    if (tid == 0) a.out_n[b] = n;
  }
  cluster.sync();  // every CTA has read the rows' records; no peer reads this CTA's shared memory
  if (lost && tid == 0) (void)mbar_wait_bounded(&sh.bar, 0u);  // (the copy lands before the memory goes away)
  if (rank == 0) {  // leave the sequence's records zeroed
    for (int i = tid; i < 2 * k + 1; i += kDrawThreads) {
      const int r = i <= k ? rt0 + i : rd0 + (i - k - 1);
      uint4* h = reinterpret_cast<uint4*>(a.hdrs + r);
      for (int w = 0; w < static_cast<int>(sizeof(RowHdr) / 16); ++w) h[w] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// ------------------------------------------------------------ launch

constexpr int kSplitMaxDevices = 64;
struct SplitLaunchCache {
  bool ready[3] = {};
  int per_sm[3] = {};
};
std::mutex g_split_mu;
SplitLaunchCache g_split_cache[kSplitMaxDevices];

template <int DT, bool HIST>
int launch_split_t(SampleArgs a, cudaStream_t st, int variant) {
  constexpr int PV = Elt<DT>::kPerVec;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kSplitMaxDevices) return cudaErrorInvalidDevice;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(g_split_mu);
    SplitLaunchCache& cc = g_split_cache[dev];
    if (!cc.ready[variant]) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cc.per_sm[variant], split_stream_kernel<DT, HIST>, kThreads, 0);
      if (e != cudaSuccess) return e;
      cc.ready[variant] = true;
    }
    per_sm = std::max(1, cc.per_sm[variant]);
  }
  const int R = a.B * (2 * a.k + 1);
  const long long nvr = a.V / PV;
  const long long units = static_cast<long long>(R) * nvr;
  // one wave; at most one CTA per 256 vectors; the piece records fit the tag area (14 R slots beyond R)
  long long g = static_cast<long long>(num_sms()) * per_sm;
  g = std::min(g, (units + 255) / 256);
  g = std::min(g, 14LL * R);
  g = std::max(1LL, g);
  a.split_grid = static_cast<int>(g);
  split_stream_kernel<DT, HIST><<<static_cast<unsigned>(g), kThreads, 0, st>>>(a);
  split_row_kernel<DT, HIST><<<static_cast<unsigned>(R), kThreads, 0, st>>>(a);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kDrawCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  const size_t dsmem = 2u * static_cast<size_t>(draw_slice_vecs(a.V / PV)) * 16u;
  e = cudaFuncSetAttribute(split_draw_kernel<DT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  if (dsmem > 48u * 1024u) {
    e = cudaFuncSetAttribute(split_draw_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dsmem));
    if (e != cudaSuccess) return e;
  }
  cfg.gridDim = dim3(static_cast<unsigned>(a.B * kDrawCl));
  cfg.blockDim = dim3(kDrawThreads);
  cfg.dynamicSmemBytes = dsmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, split_draw_kernel<DT>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// The split launch takes sampling calls (not spec_transform_probs) whose rows
// start on 16-byte boundaries and hold whole vectors; a filter needs bf16.
bool split_supported(const SampleArgs& a, int dtype) {
  if (a.mode != MODE_SAMPLE || a.k < 1) return false;
  if (!a.aligned_target || !a.aligned_draft) return false;
  const bool filt = a.top_k > 0 || a.top_p < 1.f;
  if (filt && dtype != DT_BF16) return false;
  const int pv = dtype == DT_BF16 ? 8 : 4;
  // whole vectors; the draw's two slices fit one CTA's shared memory (rows up to 512 KiB)
  return a.V % pv == 0 && a.V / pv <= 32768;
}

int launch_split(SampleArgs a, int dtype, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool filt = a.top_k > 0 || a.top_p < 1.f;
  if (dtype == DT_BF16) {
    if (filt) return launch_split_t<DT_BF16, true>(a, st, 0);
    return launch_split_t<DT_BF16, false>(a, st, 1);
  }
  return launch_split_t<DT_F32, false>(a, st, 2);
}

}  // namespace specv
