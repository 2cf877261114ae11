// row_kernel.cu -- speculative-sampling verification with one CTA per row.
//
// The method (Edge Inference Notes, post on speculative decoding and EAGLE-3,
// "The core idea: draft, then check", step 3; temperature, top-k and nucleus
// applied to both distributions as "Why it changes nothing about the output"
// states): for positions i = 0..k-1 the draft token x_i is accepted iff
// u_i q_i(x_i) < p_i(x_i); at the first rejection n one token is drawn from
// max(0, p_n - q_n) (renormalised) with u_{k+1}; if every draft is accepted
// the bonus token is drawn from p_k with u_k.
//
// Design.  CTA (b, r) owns row r of sequence b (r = 2i: target row i, r =
// 2i+1: draft row i, r = 2k: target row k), so that every reduction is
// local to one CTA.  The row streams through a ring of shared-memory stages
// filled by bulk copies (the TMA engine); the first pass reads HBM, later
// passes re-read the same bytes, which the ~300 rows in flight keep in L2.
//   pass 1  online maximum and mass Z = sum 2^(v c - m c), c = log2(e)/T,
//           per thread, combined over the CTA (and the NaN / +inf check);
//   pass 2  with a filter: a histogram over exact 16-bit bf16 keys in a
//           window below the maximum gives every group of equal values and
//           its count (its mass is count x 2^(v c - m c)).  For top-p the
//           window starts no lower than theta = (1 - top_p) Z / (2 V): the
//           tokens below theta hold less than (1 - top_p) Z, so the cut lies
//           above.  A window that does not reach the cut is followed by the
//           next one, from the largest value below it;
//   pass 3  within the group where the cut falls the lowest indices are kept
//           (rank = value descending, index ascending): the index of the
//           last kept one.
// The row's probability at the draft token follows.  The second CTA of a
// (target, draft) pair takes the accept test; the last CTA of a sequence
// finds the first rejection and draws the one token from its two rows
// (totals per chunk, then the element within the chosen chunk), writes the
// committed tokens and clears the sequence's counters.
// Sums over elements are float per thread and double-float (two floats)
// above; the kernel uses no double precision.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "device_common.cuh"
#include "internal.h"

namespace specv {
namespace {

constexpr int kStages = 4;                      // ring stages
constexpr uint32_t kStageBytes = 16384;         // bytes per stage
constexpr int kVecPerStage = kStageBytes / 16;  // 16-byte vectors per stage
constexpr int kRBins = 256;                     // exact-key histogram window (keys)
constexpr int kBinsPerThread = kRBins / kThreads;
static_assert(kBinsPerThread == 1, "one window bin per thread");
constexpr int kFirstOctaves = 12;               // top-p: the first window reaches 2^-12 of the maximum's mass
constexpr int kCandOct = 12;                    // candidates: values within 2^-12 of the running maximum's mass
constexpr int kStageCap = 128;                  // candidates a warp stages per chunk
constexpr int kCap = kRowTags / 2;              // candidates a row keeps (index + 1, bits); 0 = empty
constexpr int kSegCap = kCap / kWarps;          // a warp's own segment of the list
static_assert(kVecPerStage % kThreads == 0, "whole vectors per thread in every stage");
constexpr int kVPT = kVecPerStage / kThreads;   // vectors per thread per stage
constexpr unsigned kFullMask = 0xFFFFFFFFu;
constexpr int kMaxChunks = 64;                  // chunks the draw keeps totals for (two rows per chunk)

// A row's outcome, published in the workspace for its pair and its sequence.
struct RowOut {
  float m, c, nmc;        // maximum, log2(e)/T, -m c
  int bad;
  float zh, zl;           // Z as a double-float
  float vstar;            // kept: v > vstar, or v == vstar and index <= tie_last
  int tie_last;
  float kh, kl;           // mass of the kept set (double-float)
  float izk;              // 1 / kept mass
  float xprob;            // filtered probability at the position's draft token
  int accept;             // draft rows: the accept test of the position
  int ncand;              // candidates listed for the row (-1: the list overflowed)
  int cands_ok;           // every token of the kept set is in the list (ascending index)
  int nwritten;           // list entries written (cleared by the last user of the list)
};
static_assert(sizeof(RowOut) <= sizeof(RowHdr), "a row's outcome lives in its header slot");

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
__device__ __forceinline__ DF df_norm(DF a) {  // hi carries the rounded sum
  const float s = a.hi + a.lo;
  return DF{s, a.lo - (s - a.hi)};
}
__device__ __forceinline__ DF df_neg(DF a) { return DF{-a.hi, -a.lo}; }
__device__ __forceinline__ DF df_mulf(DF a, float f) {  // a * f, to about 2^-44
  const float p = a.hi * f;
  const float e = fmaf(a.hi, f, -p);
  return df_norm(DF{p, fmaf(a.lo, f, e)});
}
// a < b, comparing the normalised values
__device__ __forceinline__ bool df_lt(DF a, DF b) {
  const DF d = df_norm(df_add(a, df_neg(b)));
  return d.hi < 0.f;
}
__device__ __forceinline__ bool df_ge(DF a, DF b) { return !df_lt(a, b); }
__device__ __forceinline__ DF shfl_up_df(DF a, int d) {
  return DF{__shfl_up_sync(kFullMask, a.hi, d), __shfl_up_sync(kFullMask, a.lo, d)};
}
__device__ __forceinline__ DF warp_sum_dff(DF a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    DF b{__shfl_xor_sync(kFullMask, a.hi, o), __shfl_xor_sync(kFullMask, a.lo, o)};
    a = df_add(a, b);
  }
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

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
// One count into shared address addr when p holds (no branch around it).
__device__ __forceinline__ void red_shared_if(bool p, uint32_t addr) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t@q red.shared.add.u32 [%1], 1;\n\t}" ::"r"(
          static_cast<uint32_t>(p)),
      "r"(addr));
}
// Adds x to the float at shared address addr (no result, no dependency).
__device__ __forceinline__ void red_shared_f32(uint32_t addr, float x) {
  asm volatile("red.shared.add.f32 [%0], %1;" ::"r"(addr), "f"(x));
}
// Softmax mass relative to the row maximum: 2^(v c + nmc), nmc = -m c.  Every
// mass (element, histogram bin, draft token) goes through this expression.
__device__ __forceinline__ float mass(float v, float c, float nmc) { return ex2_approx(fmaf(v, c, nmc)); }
template <int DT>
__device__ __forceinline__ float val(const uint4& x, int j) {
  return Elt<DT>::value(Elt<DT>::bits_of(x, j));
}
__device__ __forceinline__ uint32_t key_of_value(float v) { return Elt<DT_BF16>::key(__float_as_uint(v) >> 16); }
__device__ __forceinline__ float value_of_key(uint32_t k) {
  return Elt<DT_BF16>::value(Elt<DT_BF16>::bits_of_key(k));
}

}  // namespace


namespace {

// ------------------------------------------------------------ the ring

struct alignas(16) RowShm {
  uint64_t full[kStages];
  uint64_t empty[kStages];  // pass 1: one arrival per warp once it has read a stage
  uint32_t gnext;          // chunks issued so far (stage = g % kStages, parity = (g / kStages) & 1)
  int timed_out;
  int stop;                // a consumer asks the stream to end after this chunk
  int withhold;            // failure-detection mode: copies withheld, waits run out
  int poll_limit;
  // per-warp partials
  float wf[kWarps][4];
  DF wd[kWarps][2];
  uint32_t wu[kWarps][2];
  // broadcast values
  float m, c, nmc;
  int bad;
  DF z;
  float vstar;
  int tie_last;
  DF zkept;
  // cut search
  int phase;               // 0 top-k, 1 top-p, 2 done
  uint32_t top_key, base_key, floor_key, first_floor;
  int floor_avail;
  uint32_t cnt_before;
  DF mass_before, target, zk;
  int gcount, gkept;
  float k_vstar;
  int k_gcount, k_gkept;
  int hit_bin;
  // ties
  int tie_target, tie_found;
  uint32_t tie_seen;
  // the draw and the sequence
  int dodraw, drawn, assemble, dchunk, dvec, dlast, retry;
  // candidates
  uint32_t mrun_key;       // running maximum over the chunks seen, as an ordered key
  int ncand, overflow, src_cands;
  uint32_t line_key;       // every token with a key at or above it is listed
  int wcnt[kWarps], wbase[kWarps];
  float dtarget;
  RowOut ro[2];            // the two rows of a draw
};

// Waits for phase `parity` of `bar` for at most `polls` polls.
__device__ __forceinline__ bool mbar_wait_polls(uint64_t* bar, uint32_t parity, int polls) {
  for (int it = 0; it < polls; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    __nanosleep(64);
  }
  return false;
}

// Bytes of a row handled per chunk: a whole stage, or half of it for each of
// two rows streamed together.
__device__ __forceinline__ uint32_t chunk_bytes(int nrows) { return nrows == 2 ? kStageBytes / 2 : kStageBytes; }

// Streams chunks [c0, c1) of one or two rows through the ring and calls
// consume(c, stage_addr, nvec) for every chunk, in order, on all threads;
// stage_addr holds the chunk (the second row's part at + kStageBytes/2).  A
// consumer that sets sh.stop ends the stream after its chunk (the copies
// already issued are waited for).  Rows that are not 16-byte aligned are
// copied with plain loads and padded with -inf.  Returns false (on every
// thread) if a copy timed out.
template <int DT, typename F>
__device__ bool stream_rows(RowShm& sh, unsigned char* ring, const unsigned char* const* rows, int nrows,
                            int V, bool aligned, int c0, int c1, F&& consume) {
  // failure-detection mode: no copy is issued and every bounded wait runs out
  const bool withhold = sh.withhold != 0;
  constexpr int E = Elt<DT>::kBytes;
  const uint32_t cb = chunk_bytes(nrows);
  const uint32_t row_bytes = static_cast<uint32_t>(V) * E;
  const int tid = threadIdx.x;
  const uint32_t g0 = sh.gnext;
  const uint32_t ring_addr = smem_addr(ring);
  auto issue = [&](int c) {  // thread 0: chunk c into its stage
    const uint32_t g = g0 + static_cast<uint32_t>(c - c0);
    const int s = static_cast<int>(g % kStages);
    const uint32_t off = static_cast<uint32_t>(c) * cb;
    const uint32_t n = min(cb, row_bytes - off);
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&sh.full[s], n * nrows);
    for (int r = 0; r < nrows; ++r)
      bulk_copy_g2s_addr(ring_addr + s * kStageBytes + r * (kStageBytes / 2), rows[r] + off, n, &sh.full[s]);
  };
  int issued = c0;  // chunks [c0, issued) are in flight or done (thread 0's count)
  if (tid == 0) {
    sh.stop = 0;
    if (aligned && !sh.timed_out && !withhold)
      for (; issued < min(c1, c0 + kStages); ++issued) issue(issued);
  }
  bool ok = !sh.timed_out;
  __syncthreads();
  int c = c0;
  for (; c < c1; ++c) {
    const uint32_t g = g0 + static_cast<uint32_t>(c - c0);
    const int s = static_cast<int>(g % kStages);
    const uint32_t off = static_cast<uint32_t>(c) * cb;
    const uint32_t n = min(cb, row_bytes - off);
    const int nvec = static_cast<int>((n + 15) / 16);
    const uint32_t st = ring_addr + s * kStageBytes;
    if (aligned) {
      if (ok && !(withhold ? mbar_wait_polls(&sh.full[s], (g / kStages) & 1u, sh.poll_limit)
                           : mbar_wait_bounded(&sh.full[s], (g / kStages) & 1u)))
        sh.timed_out = 1;
    } else {
      for (int r = 0; r < nrows; ++r) {
        const unsigned char* src = rows[r] + off;
        const uint32_t dst = st + r * (kStageBytes / 2);
        const int ne = static_cast<int>(n / E), nfill = nvec * (16 / E);
        for (int e = tid; e < nfill; e += kThreads) {
          const uint32_t bits = e < ne ? Elt<DT>::bits_at(src, e) : (E == 2 ? 0xFF80u : 0xFF800000u);
          if (E == 2) sts_u16(dst + 2u * e, bits); else sts_u32(dst + 4u * e, bits);
        }
      }
    }
    __syncthreads();
    ok = !sh.timed_out;
    if (ok) consume(c, st, nvec);
    __syncthreads();
    if (sh.stop || !ok) break;
    if (aligned && tid == 0 && c + kStages < c1 && !withhold) {
      issue(c + kStages);
      issued = c + kStages + 1;
    }
  }
  if (tid == 0) {
    // wait for copies issued past the chunk the stream ended at
    if (aligned)
      for (int c2 = c + 1; c2 < issued; ++c2) {
        const uint32_t g = g0 + static_cast<uint32_t>(c2 - c0);
        if (!mbar_wait_bounded(&sh.full[g % kStages], (g / kStages) & 1u)) sh.timed_out = 1;
      }
    sh.gnext = g0 + static_cast<uint32_t>(max(0, (aligned ? issued : c1) - c0));
    sh.stop = 0;
  }
  __syncthreads();
  return ok && !sh.timed_out;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// The first pass over one row: like stream_rows, but without CTA barriers.
// Every warp reads its own part of each stage, then arrives on the stage's
// empty barrier; thread 0 refills a stage once every warp has arrived.  The
// consumer sees only its warp's part and may use warp collectives only.
// Must start with no copy in flight (the ring's first use in the CTA).
template <int DT, typename F>
__device__ bool stream_pass1(RowShm& sh, unsigned char* ring, const unsigned char* row, int V, bool aligned,
                             int nch, F&& consume) {
  constexpr int E = Elt<DT>::kBytes;
  const uint32_t row_bytes = static_cast<uint32_t>(V) * E;
  const int tid = threadIdx.x, lane = tid & 31;
  if (!aligned || sh.withhold) {  // plain copies (or the failure-detection mode): the barrier version
    const unsigned char* rows1[1] = {row};
    return stream_rows<DT>(sh, ring, rows1, 1, V, aligned, 0, nch, consume);
  }
  const uint32_t ring_addr = smem_addr(ring);
  auto issue = [&](int c) {
    const int s = c % kStages;
    const uint32_t off = static_cast<uint32_t>(c) * kStageBytes;
    const uint32_t n = min(kStageBytes, row_bytes - off);
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&sh.full[s], n);
    bulk_copy_g2s_addr(ring_addr + s * kStageBytes, row + off, n, &sh.full[s]);
  };
  int issued = 0;  // thread 0's count of chunks issued
  if (tid == 0)
    for (; issued < min(nch, kStages); ++issued) issue(issued);
  bool ok = true;
  for (int c = 0; c < nch; ++c) {
    const int s = c % kStages;
    const uint32_t par = static_cast<uint32_t>(c / kStages) & 1u;
    if (tid == 0 && c >= 1 && c - 1 + kStages < nch && ok) {
      // refill the stage of chunk c - 1 once every warp has read it
      const int sp = (c - 1) % kStages;
      if (mbar_wait_bounded(&sh.empty[sp], static_cast<uint32_t>((c - 1) / kStages) & 1u)) {
        issue(c - 1 + kStages);
        issued = c + kStages;
      } else {
        ok = false;
      }
    }
    if (ok && !mbar_wait_bounded(&sh.full[s], par)) ok = false;
    ok = __shfl_sync(kFullMask, ok ? 1 : 0, 0) != 0 && __all_sync(kFullMask, ok);
    if (!ok) break;
    const uint32_t off = static_cast<uint32_t>(c) * kStageBytes;
    const int nvec = static_cast<int>((min(kStageBytes, row_bytes - off) + 15) / 16);
    consume(c, ring_addr + s * kStageBytes, nvec);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
  }
  if (!ok) sh.timed_out = 1;
  __syncthreads();
  if (tid == 0) sh.gnext = static_cast<uint32_t>(issued);  // (on a timeout, drain_ring waits for these)
  __syncthreads();
  return !sh.timed_out;
}

// A CTA whose copies timed out waits (bounded) for the last copy issued to
// every stage before its shared memory goes away.
__device__ void drain_ring(RowShm& sh) {
  if (threadIdx.x != 0 || !sh.timed_out || sh.withhold) return;
  const uint32_t g = sh.gnext;
  for (int d = 1; d <= kStages && static_cast<uint32_t>(d) <= g; ++d) {
    const uint32_t gl = g - d;
    (void)mbar_wait_bounded(&sh.full[gl % kStages], (gl / kStages) & 1u);
  }
}

// CTA sum of one double-float per thread (thread order within warps, then
// warps in order); the result on every thread.
__device__ DF cta_sum_df(RowShm& sh, DF v, int slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_dff(v);
  if (lane == 0) sh.wd[warp][slot] = v;
  __syncthreads();
  DF t = df_make(0.f);
  for (int w = 0; w < kWarps; ++w) t = df_add(t, sh.wd[w][slot]);
  __syncthreads();
  return df_norm(t);
}

}  // namespace

// ------------------------------------------------------------ the draw

namespace {

// The draw of one token by inverse CDF in ascending index order, over the
// rows ro[0] (target) and, for a residual, ro[1] (draft): mode 0 weights
// max(0, p - q), mode 1 weights p; a residual of mass zero falls back to p.
// Totals per chunk first, then the element within the chunk that holds
// u * S.  Returns the token (on every thread), or -1.
template <int DT>
__device__ int draw_token(RowShm& sh, unsigned char* ring, DF* ctot, const unsigned char* trow,
                          const unsigned char* drow, int V, bool aligned, float u) {
  constexpr int E = Elt<DT>::kBytes;
  constexpr int PV = Elt<DT>::kPerVec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool pair = drow != nullptr;
  const unsigned char* rows[2] = {trow, drow};
  const int nr = pair ? 2 : 1;
  const int cb = static_cast<int>(chunk_bytes(nr));
  const int nch = static_cast<int>((static_cast<uint32_t>(V) * E + cb - 1) / cb);
  const int epc = cb / E;
  const float cp = sh.ro[0].c, np = sh.ro[0].nmc, vsp = sh.ro[0].vstar, ip = sh.ro[0].izk;
  const int tlp = sh.ro[0].tie_last;
  const float cq = sh.ro[1].c, nq = sh.ro[1].nmc, vsq = sh.ro[1].vstar, iq = sh.ro[1].izk;
  const int tlq = sh.ro[1].tie_last;
  auto weights = [&](int mode, uint32_t st, int v, int t0, float* w) {
    const uint4 qp = lds128(st + 16u * v);
    uint4 qq = qp;
    if (mode == 0) qq = lds128(st + kStageBytes / 2 + 16u * v);
#pragma unroll
    for (int jj = 0; jj < PV; ++jj) {
      const int t = t0 + jj;
      const float lp = val<DT>(qp, jj);
      float wt = (lp > vsp || (lp == vsp && t <= tlp)) ? mass(lp, cp, np) * ip : 0.f;
      if (mode == 0) {
        const float lq = val<DT>(qq, jj);
        const float wq = (lq > vsq || (lq == vsq && t <= tlq)) ? mass(lq, cq, nq) * iq : 0.f;
        wt = fmaxf(wt - wq, 0.f);
      }
      w[jj] = wt;
    }
  };
  if (tid == 0) sh.drawn = -1;
  for (int mode = pair ? 0 : 1; mode < 2; ++mode) {
    // totals per chunk (per warp in shared memory, no CTA barrier per chunk)
    bool ok = stream_rows<DT>(sh, ring, rows, nr, V, aligned, 0, nch, [&](int ch, uint32_t st, int nvec) {
      float part = 0.f;
#pragma unroll
      for (int j = 0; j < kVPT; ++j) {
        const int v = tid + j * kThreads;
        if (v >= nvec) break;
        float w[PV];
        weights(mode, st, v, ch * epc + v * PV, w);
#pragma unroll
        for (int jj = 0; jj < PV; ++jj) part += w[jj];
      }
      DF t = warp_sum_dff(df_make(part));
      if (lane == 0) ctot[ch * kWarps + warp] = t;
    });
    if (!ok) return -1;
    if (tid == 0) {
      DF S = df_make(0.f);
      for (int e = 0; e < nch * kWarps; ++e) S = df_add(S, ctot[e]);
      S = df_norm(S);
      sh.retry = mode == 0 && !(S.hi > 0.f);
      if (!sh.retry) {
        const DF tgt = df_mulf(S, u);
        int pick = -1;
        DF cum = df_make(0.f);
        for (int ch = 0; ch < nch && pick < 0; ++ch) {
          DF t = df_make(0.f);
          for (int w = 0; w < kWarps; ++w) t = df_add(t, ctot[ch * kWarps + w]);
          const DF nx = df_add(cum, t);
          if (t.hi > 0.f && df_lt(tgt, nx)) pick = ch;
          else cum = nx;
        }
        if (pick < 0) {  // rounding: the last chunk with mass
          cum = df_make(0.f);
          for (int ch = 0; ch < nch; ++ch) {
            DF t = df_make(0.f);
            for (int w = 0; w < kWarps; ++w) t = df_add(t, ctot[ch * kWarps + w]);
            if (t.hi > 0.f) pick = ch;
          }
          for (int e = 0; e < pick * kWarps; ++e) cum = df_add(cum, ctot[e]);
        }
        const DF rem = df_norm(df_add(tgt, df_neg(cum)));
        sh.dchunk = pick;
        sh.dtarget = rem.hi + rem.lo;
        sh.dvec = 0x7FFFFFFF;
        sh.dlast = -1;
      }
    }
    __syncthreads();
    if (sh.retry) continue;  // a residual of mass zero: draw from p
    const int pick = sh.dchunk;
    if (pick < 0) return -1;
    ok = stream_rows<DT>(sh, ring, rows, nr, V, aligned, pick, pick + 1, [&](int ch, uint32_t st, int nvec) {
      float base = 0.f;
      const float tw = sh.dtarget;
      for (int j = 0; j < kVPT; ++j) {
        const int v = tid + j * kThreads;
        float w[PV];
        float ls = 0.f;
        if (v < nvec) {
          weights(mode, st, v, ch * epc + v * PV, w);
#pragma unroll
          for (int jj = 0; jj < PV; ++jj) ls += w[jj];
        } else {
#pragma unroll
          for (int jj = 0; jj < PV; ++jj) w[jj] = 0.f;
        }
        float incl = ls;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(kFullMask, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane == 31) sh.wf[warp][3] = incl;
        __syncthreads();
        float pre = 0.f, rt = 0.f;
        for (int w2 = 0; w2 < kWarps; ++w2) {
          if (w2 < warp) pre += sh.wf[w2][3];
          rt += sh.wf[w2][3];
        }
        incl += pre;
        if (ls > 0.f) {
          atomicMax(&sh.dlast, v);
          if (base + incl > tw) atomicMin(&sh.dvec, v);
        }
        __syncthreads();
        if (sh.dvec != 0x7FFFFFFF) {
          if (v == sh.dvec) {  // the element within the vector
            const float t0 = tw - (base + incl - ls);
            float acc = 0.f;
            int jj = -1, lj = -1;
            for (int q = 0; q < PV; ++q) {
              if (w[q] > 0.f) lj = q;
              acc += w[q];
              if (jj < 0 && w[q] > 0.f && acc > t0) jj = q;
            }
            sh.drawn = ch * epc + v * PV + (jj >= 0 ? jj : lj);
          }
          break;
        }
        base += rt;
        __syncthreads();
      }
      __syncthreads();
      if (sh.drawn < 0 && sh.dlast >= 0 && tid == (sh.dlast % kThreads)) {
        // rounding left the target past the chunk: its last element with weight
        const int v = sh.dlast;
        float w[PV];
        weights(mode, st, v, ch * epc + v * PV, w);
        int lj = 0;
        for (int q = 0; q < PV; ++q)
          if (w[q] > 0.f) lj = q;
        sh.drawn = ch * epc + v * PV + lj;
      }
    });
    if (!ok) return -1;
    break;
  }
  __syncthreads();
  return sh.drawn;
}

}  // namespace

// ------------------------------------------------------------ candidates

namespace {

__device__ __forceinline__ uint32_t f32_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float f32_of_key(uint32_t k) {
  if (k == 0u) return -INFINITY;
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Appends this warp's elements of a staged chunk at or above vth to its
// own segment of the row's list (wc: the warp's count, the same in every
// lane), as (index + 1, bits); a full segment sets the row's overflow flag.
template <int DT>
__device__ __forceinline__ void append_candidates(RowShm& sh, uint32_t st, int nvec, int ch, int epc, float vth,
                                                  uint2* list, int& wc) {
  constexpr int PV = Elt<DT>::kPerVec;
  constexpr int kWarpVecs = kVecPerStage / kWarps;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint2* seg = list + warp * kSegCap;
#pragma unroll
  for (int j = 0; j < kVPT; ++j) {
    const int v = warp * kWarpVecs + j * 32 + lane;
    uint32_t msk = 0;
    uint4 q = make_uint4(0, 0, 0, 0);
    if (v < nvec) {
      q = lds128(st + 16u * v);
#pragma unroll
      for (int jj = 0; jj < PV; ++jj) msk |= (val<DT>(q, jj) >= vth ? 1u : 0u) << jj;
    }
    if (!__ballot_sync(kFullMask, msk != 0u)) continue;
    const int cn = __popc(msk);
    int ex = cn;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFullMask, ex, o);
      if (lane >= o) ex += y;
    }
    const int tot = __shfl_sync(kFullMask, ex, 31);
    ex -= cn;
    if (wc + tot > kSegCap) {
      sh.overflow = 1;
      wc = kSegCap;
      return;
    }
    int pos = wc + ex;
    if (msk) {
#pragma unroll
      for (int jj = 0; jj < PV; ++jj)
        if (msk >> jj & 1u)
          seg[pos++] = make_uint2(static_cast<uint32_t>(ch * epc + v * PV + jj) + 1u, Elt<DT>::bits_of(q, jj));
    }
    wc += tot;
  }
}

}  // namespace

// ------------------------------------------------------------ the draw over candidates

namespace {

// Ascending bitonic sort of n (a power of two) keys in shared memory, by
// the whole CTA.
template <typename K>
__device__ void bitonic_sort(K* a, int n) {
  for (int size = 2; size <= n; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < n / 2; t += kThreads) {
        const int i0 = 2 * stride * (t / stride) + (t % stride);
        const int i1 = i0 + stride;
        const bool up = (i0 & size) == 0;
        const K x = a[i0], y = a[i1];
        if ((x > y) == up) {
          a[i0] = y;
          a[i1] = x;
        }
      }
      __syncthreads();
    }
}

// The draw over a target row's kept tokens, sorted by index as
// (index << 32 | value bits): weights max(0, p - q) (q read from the
// draft row at the listed tokens) or, without a draft row (or for a residual
// of mass zero), p.  Rounds of kThreads entries: totals per round, then the
// entry within the round whose running total passes u * S.  Returns the
// token (on every thread), or -1.
template <int DT>
__device__ int draw_cands(RowShm& sh, DF* ctot, const unsigned long long* list, int n, const unsigned char* drow,
                          float u) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float cp = sh.ro[0].c, np = sh.ro[0].nmc, vsp = sh.ro[0].vstar, ip = sh.ro[0].izk;
  const int tlp = sh.ro[0].tie_last;
  const float cq = sh.ro[1].c, nq = sh.ro[1].nmc, vsq = sh.ro[1].vstar, iq = sh.ro[1].izk;
  const int tlq = sh.ro[1].tie_last;
  auto weight = [&](int mode, int e, int* tok) -> float {
    *tok = -1;
    if (e >= n) return 0.f;
    const unsigned long long en = list[e];
    const int t = static_cast<int>(en >> 32);
    *tok = t;
    const float lp = Elt<DT>::value(static_cast<uint32_t>(en));
    const float p = (lp > vsp || (lp == vsp && t <= tlp)) ? mass(lp, cp, np) * ip : 0.f;
    if (mode == 1 || p == 0.f) return p;
    const float lq = Elt<DT>::value(Elt<DT>::bits_at(drow, t));
    const float q = (lq > vsq || (lq == vsq && t <= tlq)) ? mass(lq, cq, nq) * iq : 0.f;
    return fmaxf(p - q, 0.f);
  };
  const int nr = (n + kThreads - 1) / kThreads;
  int token = -1;
  for (int mode = drow ? 0 : 1; mode < 2; ++mode) {
    for (int rd = 0; rd < nr; ++rd) {
      int t;
      const float w = weight(mode, rd * kThreads + tid, &t);
      const DF s = cta_sum_df(sh, df_make(w), 1);
      if (tid == 0) ctot[rd] = s;
    }
    __syncthreads();
    if (tid == 0) {
      DF S = df_make(0.f);
      for (int rd = 0; rd < nr; ++rd) S = df_add(S, ctot[rd]);
      S = df_norm(S);
      sh.retry = mode == 0 && !(S.hi > 0.f);
      sh.dchunk = -1;
      if (!sh.retry && S.hi > 0.f) {
        const DF tgt = df_mulf(S, u);
        DF cum = df_make(0.f);
        int pick = -1;
        for (int rd = 0; rd < nr && pick < 0; ++rd) {
          const DF nx = df_add(cum, ctot[rd]);
          if (ctot[rd].hi > 0.f && df_lt(tgt, nx)) pick = rd;
          else cum = nx;
        }
        if (pick < 0) {  // rounding: the last round with mass
          cum = df_make(0.f);
          for (int rd = 0; rd < nr; ++rd)
            if (ctot[rd].hi > 0.f) pick = rd;
          for (int rd = 0; rd < pick; ++rd) cum = df_add(cum, ctot[rd]);
        }
        const DF rem = df_norm(df_add(tgt, df_neg(cum)));
        sh.dchunk = pick;
        sh.dtarget = rem.hi + rem.lo;
      }
      sh.dvec = 0x7FFFFFFF;
      sh.dlast = -1;
    }
    __syncthreads();
    if (sh.retry) continue;
    const int rd = sh.dchunk;
    if (rd < 0) break;
    int t;
    const float w = weight(mode, rd * kThreads + tid, &t);
    float incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.wf[warp][3] = incl;
    __syncthreads();
    float pre = 0.f;
    for (int w2 = 0; w2 < warp; ++w2) pre += sh.wf[w2][3];
    incl += pre;
    if (w > 0.f) {
      atomicMax(&sh.dlast, tid);
      if (incl > sh.dtarget) atomicMin(&sh.dvec, tid);
    }
    __syncthreads();
    const int pickt = sh.dvec != 0x7FFFFFFF ? sh.dvec : sh.dlast;
    if (tid == pickt) sh.drawn = t;
    __syncthreads();
    if (pickt >= 0) token = sh.drawn;
    break;
  }
  __syncthreads();
  return token;
}

}  // namespace

// ------------------------------------------------------------ the kernel

template <int DT, bool FILTER>
__global__ void __launch_bounds__(kThreads, 2) row_kernel(SampleArgs a) {
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ RowShm sh;
  // window counts, one private copy per warp lane: [bin][lane], so that no
  // two lanes of a warp ever add to the same word
  __shared__ __align__(16) uint32_t hist[FILTER ? kRBins * 32 : 1];
  __shared__ DF ctot[kMaxChunks * kWarps];
  constexpr int E = Elt<DT>::kBytes;
  constexpr int PV = Elt<DT>::kPerVec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = a.B, k = a.k, V = a.V;
  const int R = 2 * k + 1;
  // position-major: every sequence's rows of position 0 first, so that a
  // position's predecessors have usually finished when it decides
  const int r = blockIdx.x / B, b = blockIdx.x % B;
  const bool is_target = (r & 1) == 0;
  const int i = r / 2;  // position (k for the bonus row)
  RowOut* outs = reinterpret_cast<RowOut*>(a.hdrs);
  RowOut* me = outs + static_cast<size_t>(b) * R + r;
  uint2* lists = reinterpret_cast<uint2*>(a.tags);
  uint2* mylist = lists + (static_cast<size_t>(b) * R + r) * kCap;
  const unsigned char* trow_base = static_cast<const unsigned char*>(a.target);
  const unsigned char* drow_base = static_cast<const unsigned char*>(a.draft);
  const unsigned char* row = is_target ? trow_base + (static_cast<size_t>(b) * (k + 1) + i) * V * E
                                       : drow_base + (static_cast<size_t>(b) * k + i) * V * E;
  const bool aligned = is_target ? a.aligned_target : a.aligned_draft;
  const int nchunks = static_cast<int>((static_cast<uint32_t>(V) * E + kStageBytes - 1) / kStageBytes);
  const int epc = static_cast<int>(kStageBytes) / E;  // elements per chunk (one row)
  volatile uint32_t* rej_word = a.draw_tickets + b;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kWarps);
    }
    fence_mbar_init();
    sh.gnext = 0;
    sh.timed_out = 0;
    sh.stop = 0;
    sh.withhold = a.launch_mode == SPEC_LAUNCH_FUSED_WAIT_TEST;
    sh.poll_limit = a.poll_limit;
    sh.assemble = 0;
    sh.dodraw = 0;
    sh.drawn = -1;
    sh.mrun_key = 0u;
    sh.ncand = 0;
    sh.overflow = 0;
    sh.src_cands = 0;
    sh.line_key = 0xFFFFFFFFu;
  }
  // the draft token's value in this row, read early
  int x = -1;
  float xv = 0.f;
  if (tid == 0 && i < k) {
    x = a.tokens[static_cast<size_t>(b) * k + i];
    if (x >= 0 && x < V) xv = Elt<DT>::value(Elt<DT>::bits_at(row, x));
  }
  const float T = a.temperature_per_seq ? a.temperature_per_seq[b] : a.temperature;
  const bool t_ok = T > 0.f && isfinite(T);
  const float c = t_ok ? kLog2e / T : 0.f;
  // candidates lie within kCandOct octaves of mass (and a little more) below the running maximum
  const float cand_span = t_ok ? (static_cast<float>(kCandOct) + 0.01f) / c : 0.f;
  __syncthreads();

  // ---- pass 1: online maximum and mass per thread; with a filter, the
  // candidates, appended in ascending index
  float mt = -INFINITY, nmct = 0.f;
  DF zt = df_make(0.f);
  uint32_t nanacc = 0xFF80FF80u;  // bf16: NaN-propagating maximum of everything
  float nanf = -INFINITY;
  const unsigned char* rows1[1] = {row};
  constexpr int kWarpVecs = kVecPerStage / kWarps;  // a warp's contiguous vectors in a chunk
  int wcand = 0;          // this warp's candidates (the same in every lane)
  float wrun = -INFINITY;  // this warp's running maximum over the chunks before
  bool ok = stream_pass1<DT>(sh, ring, row, V, aligned, nchunks, [&](int ch, uint32_t st, int nvec) {
    // this lane's vectors of the chunk, loaded first (past the row's end: -inf)
    uint4 q[kVPT];
#pragma unroll
    for (int j = 0; j < kVPT; ++j) {
      const int v = warp * kWarpVecs + j * 32 + lane;
      q[j] = v < nvec ? lds128(st + 16u * v)
                      : (DT == DT_BF16 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                       : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u));
    }
    // the lane's maximum over them (NaN-propagating for the check), one rescale per chunk
    float cmax;
    if (DT == DT_BF16) {
      uint32_t m2 = 0xFF80FF80u;
#pragma unroll
      for (int j = 0; j < kVPT; ++j) m2 = bmax2_nan(m2, bmax2_nan(bmax2_nan(q[j].x, q[j].y), bmax2_nan(q[j].z, q[j].w)));
      nanacc = bmax2_nan(nanacc, m2);
      cmax = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
    } else {
      float m1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < kVPT; ++j)
        m1 = fmax_nan(m1, fmax_nan(fmax_nan(__uint_as_float(q[j].x), __uint_as_float(q[j].y)),
                                   fmax_nan(__uint_as_float(q[j].z), __uint_as_float(q[j].w))));
      nanf = fmax_nan(nanf, m1);
      cmax = m1;
    }
    if (cmax > mt) {  // a new maximum: rescale what this thread has summed
      if (mt > -INFINITY) zt = df_mulf(zt, ex2_approx((mt - cmax) * c));
      mt = cmax;
      nmct = -cmax * c;
    }
    float p0 = 0.f, p1 = 0.f;
#pragma unroll
    for (int j = 0; j < kVPT; ++j) {
      float e[PV];
#pragma unroll
      for (int jj = 0; jj < PV; ++jj) e[jj] = mass(val<DT>(q[j], jj), c, nmct);
      p0 += (e[0] + e[1 % PV]) + (e[2 % PV] + e[3 % PV]);
      if (PV == 8) p1 += (e[4 % PV] + e[5 % PV]) + (e[6 % PV] + e[7 % PV]);
    }
    zt = df_add(zt, p0 + p1);
    if constexpr (FILTER) {
      // candidates of this chunk: at or above the running maximum (the CTA's,
      // kept with atomicMax, never above the row's) less the span; chunk 0 is
      // listed after the pass, with the row's maximum
      const bool on = ch > 0 && __shfl_sync(kFullMask, sh.overflow, 0) == 0;
      const float th = fmaxf(wrun, f32_of_key(sh.mrun_key)) - cand_span;
      float wm = cmax;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(kFullMask, wm, o));
      if (lane == 0 && wm > -INFINITY) atomicMax(&sh.mrun_key, f32_key(wm));
      wrun = fmaxf(wrun, wm);
      if (on) {
        uint32_t tb = __float_as_uint(th) & 0xFFFF0000u;  // the threshold rounded down to bf16, in both halves
        if (__uint_as_float(tb) > th) tb += 0x10000u;
        if (!(th > -INFINITY)) tb = 0xFF800000u;
        const uint32_t t2u = (tb >> 16) | tb;
        const __nv_bfloat162 t2 = *reinterpret_cast<const __nv_bfloat162*>(&t2u);
        uint32_t vmask = 0;  // a bit per vector holding a candidate
#pragma unroll
        for (int j = 0; j < kVPT; ++j) {
          const uint32_t g = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&q[j].x), t2) |
                             __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&q[j].y), t2) |
                             __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&q[j].z), t2) |
                             __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&q[j].w), t2);
          vmask |= (g != 0u && warp * kWarpVecs + j * 32 + lane < nvec ? 1u : 0u) << j;
        }
        if (__ballot_sync(kFullMask, vmask != 0u)) {
          // the flagged vectors' elements (work in proportion to what is flagged),
          // then one warp scan for the chunk
          auto pick = [&](int j) -> uint4 { return j == 0 ? q[0] : (j == 1 ? q[1] : (j == 2 ? q[2] : q[3])); };
          uint32_t cmask = 0;
          for (uint32_t vm = vmask; vm; vm &= vm - 1u) {
            const int j = __ffs(vm) - 1;
            const uint4 qq = pick(j);
            const uint32_t g0 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&qq.x), t2);
            const uint32_t g1 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&qq.y), t2);
            const uint32_t g2 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&qq.z), t2);
            const uint32_t g3 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&qq.w), t2);
            const uint32_t bits8 = (g0 & 1u) | ((g0 >> 15) & 2u) | ((g1 & 1u) << 2) | ((g1 >> 13) & 8u) |
                                   ((g2 & 1u) << 4) | ((g2 >> 11) & 32u) | ((g3 & 1u) << 6) | ((g3 >> 9) & 128u);
            cmask |= bits8 << (8 * j);
          }
          const int cn = __popc(cmask);
          int ex = cn;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFullMask, ex, o);
            if (lane >= o) ex += y;
          }
          const int tot = __shfl_sync(kFullMask, ex, 31);
          ex -= cn;
          if (wcand + tot > kSegCap) {
            if (lane == 0) sh.overflow = 1;
          } else {
            uint2* seg = mylist + warp * kSegCap + wcand + ex;
            for (uint32_t cm = cmask; cm; cm &= cm - 1u) {
              const int bit = __ffs(cm) - 1;
              const int j = bit >> 3, jj = bit & 7;
              const uint4 qq = pick(j);
              const uint32_t w = (jj >> 1) == 0 ? qq.x : ((jj >> 1) == 1 ? qq.y : ((jj >> 1) == 2 ? qq.z : qq.w));
              const uint32_t bits = (jj & 1) ? (w >> 16) : (w & 0xFFFFu);
              const int v = warp * kWarpVecs + j * 32 + lane;
              *seg++ = make_uint2(static_cast<uint32_t>(ch * epc + v * PV + jj) + 1u, bits);
            }
            wcand += tot;
          }
        }
      }
    }
  });
  // combine over the CTA: m = max, Z = sum z_t 2^((m_t - m) c)
  {
    float bad_t = 0.f;
    if (DT == DT_BF16) {
      const float n0 = fmax_nan(__uint_as_float(nanacc << 16), __uint_as_float(nanacc & 0xFFFF0000u));
      bad_t = (n0 != n0 || n0 == INFINITY) ? 1.f : 0.f;
    } else {
      bad_t = (nanf != nanf || nanf == INFINITY) ? 1.f : 0.f;
    }
    float wm = mt;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(kFullMask, wm, o));
    const float wb = __reduce_max_sync(kFullMask, static_cast<unsigned>(bad_t)) ? 1.f : 0.f;
    if (lane == 0) {
      sh.wf[warp][0] = wm;
      sh.wf[warp][1] = wb;
    }
    __syncthreads();
    float m = -INFINITY, bad = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      m = fmaxf(m, sh.wf[w][0]);
      bad = fmaxf(bad, sh.wf[w][1]);
    }
    __syncthreads();
    const bool row_bad = !ok || bad != 0.f || !t_ok || !(m > -INFINITY) || !(m < INFINITY);
    DF zs = df_make(0.f);
    if (!row_bad && mt > -INFINITY) zs = df_mulf(zt, ex2_approx((mt - m) * c));
    const DF Z = cta_sum_df(sh, zs, 0);
    if (tid == 0) {
      sh.m = m;
      sh.c = c;
      sh.nmc = row_bad ? 0.f : -m * c;
      sh.bad = row_bad;
      sh.z = Z;
      sh.vstar = -INFINITY;
      sh.tie_last = 0x7FFFFFFF;
      sh.zkept = Z;
    }
    __syncthreads();
  }

  // ---- the cut
  if constexpr (FILTER) {
    if (!sh.bad && !sh.overflow) {  // chunk 0, listed now with the row's maximum (from L2)
      const float vth0 = sh.m - cand_span;
      ok = stream_rows<DT>(sh, ring, rows1, 1, V, aligned, 0, min(1, nchunks), [&](int ch, uint32_t st, int nvec) {
        append_candidates<DT>(sh, st, nvec, ch, epc, vth0, mylist, wcand);
      });
    }
    if (lane == 0) sh.wcnt[warp] = wcand;
    __syncthreads();
    if (tid == 0) {
      int t = 0;
      for (int w = 0; w < kWarps; ++w) t += sh.wcnt[w];
      sh.ncand = t;
    }
    __syncthreads();
    const int top_k = a.top_k;
    const float top_p = a.top_p;
    // lowest key a top-p window needs (see the file comment)
    auto theta_key = [&]() -> uint32_t {
      const float th = 0.5f * (1.f - top_p) * (sh.zk.hi + sh.zk.lo) / static_cast<float>(V);
      if (!(th > 0.f)) return 0u;
      const float vth = (log2f(th) - sh.nmc) / sh.c;
      if (!(vth > -INFINITY) || !(vth < INFINITY)) return 0u;
      const uint32_t bits = __float_as_uint(vth) & 0xFFFF0000u;  // toward zero
      float vb = __uint_as_float(bits);
      if (vb > vth) vb = __uint_as_float(bits + 0x10000u);       // negative: one step further down
      if (!(vb <= vth)) return 0u;
      return key_of_value(vb);
    };
    auto start_window = [&]() {  // thread 0
      uint32_t lowest = sh.top_key >= static_cast<uint32_t>(kRBins - 1) ? sh.top_key - (kRBins - 1) : 0u;
      if (sh.phase == 1) {
        uint32_t th = theta_key();
        if (sh.first_floor > th) th = sh.first_floor;  // (only for the first window)
        sh.first_floor = 0;
        if (th > lowest && th <= sh.top_key) lowest = th;
      }
      if (sh.floor_key > lowest) lowest = sh.floor_key;
      if (sh.src_cands && sh.line_key > lowest) lowest = sh.line_key;  // the list is complete down to here
      sh.base_key = lowest;
    };
    auto reset_search = [&]() {  // thread 0: the search from the top
      sh.phase = sh.bad ? 2 : (top_k > 0 ? 0 : 1);
      sh.top_key = key_of_value(sh.m);
      sh.floor_key = 0;
      sh.first_floor = 0;
      sh.floor_avail = 0;
      sh.cnt_before = 0;
      sh.mass_before = df_make(0.f);
      sh.zk = sh.z;
      sh.target = df_mulf(sh.z, top_p);
      sh.gcount = sh.gkept = 0;
      sh.k_vstar = -INFINITY;
      sh.k_gcount = sh.k_gkept = 0;
      if (sh.phase == 1) {  // the first window reaches kFirstOctaves octaves of mass below the maximum
        const float vf = (-static_cast<float>(kFirstOctaves) - sh.nmc) / sh.c;
        const uint32_t bits = __float_as_uint(vf) & 0xFFFF0000u;
        float vb = __uint_as_float(bits);
        if (vb > vf) vb = __uint_as_float(bits + 0x10000u);
        sh.first_floor = (vb <= vf && vb > -INFINITY) ? key_of_value(vb) : 0u;
      }
      if (sh.phase < 2) start_window();
    };
    if (tid == 0) {
      // candidates: every token with a value at or above m - cand_span is listed
      sh.src_cands = 0;
      if (!sh.bad && !sh.overflow) {
        const float vl = sh.m - cand_span;
        const uint32_t bits = __float_as_uint(vl) & 0xFFFF0000u;  // toward zero
        float vb = __uint_as_float(bits);
        if (vb < vl) vb = __uint_as_float(bits + 0x10000u);      // positive: one step up
        if (vb >= vl && vb <= sh.m) {
          sh.line_key = key_of_value(vb);
          sh.src_cands = 1;
        }
      }
      reset_search();
    }
    __syncthreads();
    for (int iter = 0; iter < 80 && sh.phase < 2; ++iter) {
      for (int e = tid; e < kRBins * 32; e += kThreads) hist[e] = 0u;
      const float wlo = value_of_key(sh.base_key), whi = value_of_key(sh.top_key);
      const uint32_t base = sh.base_key;
      const uint32_t haddr = smem_addr(hist);
      float bl = -INFINITY;
      __syncthreads();
      if (sh.src_cands) {
        for (int e = tid; e < kCap; e += kThreads) {
          if ((e & (kSegCap - 1)) >= sh.wcnt[e / kSegCap]) continue;
          const float f = Elt<DT>::value(mylist[e].y);
          const bool in = f >= wlo && f <= whi;
          red_shared_if(in, haddr + 4u * ((((key_of_value(f) - base) & (kRBins - 1)) << 5) | lane));
          bl = fmaxf(bl, f < wlo ? f : -INFINITY);
        }
        __syncthreads();
      } else
      ok = stream_rows<DT>(sh, ring, rows1, 1, V, aligned, 0, nchunks, [&](int, uint32_t st, int nvec) {
#pragma unroll
        for (int j = 0; j < kVPT; ++j) {
          const int v = tid + j * kThreads;
          if (v >= nvec) break;
          const uint4 q = lds128(st + 16u * v);
#pragma unroll
          for (int jj = 0; jj < PV; ++jj) {
            const float f = val<DT>(q, jj);
            if (f >= wlo && f <= whi) red_shared_if(true, haddr + 4u * ((((key_of_value(f) - base) & (kRBins - 1)) << 5) | lane));
            bl = fmaxf(bl, f < wlo ? f : -INFINITY);
          }
        }
      });
      // the group: thread t takes bins 2047-8t .. 2040-8t (keys descending)
      uint32_t cnt[kBinsPerThread];
      float mf[kBinsPerThread];
      uint32_t tc = 0;
      DF tm = df_make(0.f);
      const uint32_t top = sh.top_key, flo = sh.floor_key;
      const int favail = sh.floor_avail;
#pragma unroll
      for (int j = 0; j < kBinsPerThread; ++j) {
        const int bin = kRBins - 1 - (kBinsPerThread * tid + j);
        const uint32_t key = base + static_cast<uint32_t>(bin);
        uint32_t n = 0;
#pragma unroll 8
        for (int l = 0; l < 32; ++l) n += hist[(bin << 5) | ((l + bin) & 31)];
        if (key > top || key < flo) n = 0;  // outside the window or the top-k set
        if (flo != 0 && key == flo && n > static_cast<uint32_t>(favail)) n = static_cast<uint32_t>(favail);
        cnt[j] = n;
        mf[j] = n ? static_cast<float>(n) * mass(value_of_key(key), sh.c, sh.nmc) : 0.f;
        tc += n;
        tm = df_add(tm, mf[j]);
      }
      // exclusive scans over threads (warp scans, then warp totals in order)
      uint32_t ci = tc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFullMask, ci, o);
        if (lane >= o) ci += y;
      }
      const DF mi = warp_incl_scan_df(tm);
      if (lane == 31) {
        sh.wu[warp][0] = ci;
        sh.wd[warp][0] = mi;
      }
      float blw = bl;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) blw = fmaxf(blw, __shfl_xor_sync(kFullMask, blw, o));
      if (lane == 0) sh.wf[warp][2] = blw;
      if (tid == 0) sh.hit_bin = 0x7FFFFFFF;
      __syncthreads();
      uint32_t cpre = 0;
      DF mpre = df_make(0.f);
      for (int w = 0; w < warp; ++w) {
        cpre += sh.wu[w][0];
        mpre = df_add(mpre, sh.wd[w][0]);
      }
      uint32_t ce = __shfl_up_sync(kFullMask, ci, 1);
      DF me = shfl_up_df(mi, 1);
      if (lane == 0) {
        ce = 0;
        me = df_make(0.f);
      }
      ce += cpre + sh.cnt_before;
      me = df_add(df_add(me, mpre), sh.mass_before);
      // the first bin (from the top) whose running total reaches the target
      {
        uint32_t cc = ce;
        DF mc = me;
        const int ph = sh.phase;
        const DF tgt = sh.target;
        for (int j = 0; j < kBinsPerThread; ++j) {
          cc += cnt[j];
          mc = df_add(mc, mf[j]);
          if (cnt[j] == 0) continue;
          const bool hit = ph == 0 ? cc >= static_cast<uint32_t>(top_k) : df_ge(mc, tgt);
          if (hit) {
            atomicMin(&sh.hit_bin, kBinsPerThread * tid + j);
            break;
          }
        }
      }
      __syncthreads();
      const int hb = sh.hit_bin;
      // the owner of the hit bin (or thread kThreads-1 for the window totals) reports
      const int owner = hb != 0x7FFFFFFF ? hb / kBinsPerThread : kThreads - 1;
      if (tid == owner) {
        uint32_t cc = ce;
        DF mc = me;
        const int jh = hb != 0x7FFFFFFF ? hb % kBinsPerThread : kBinsPerThread;
        for (int j = 0; j < jh; ++j) {
          cc += cnt[j];
          mc = df_add(mc, mf[j]);
        }
        if (hb != 0x7FFFFFFF) {
          // the group found: its key, count and what lies above it
          const uint32_t gkey = base + static_cast<uint32_t>(kRBins - 1 - hb);
          uint32_t gc = 0;
          for (int j = 0; j < kBinsPerThread; ++j)
            if (j == jh) gc = cnt[j];
          const float gv = value_of_key(gkey);
          const float gw = mass(gv, sh.c, sh.nmc);
          int kept;
          if (sh.phase == 0) {
            kept = top_k - static_cast<int>(cc);
          } else {
            const DF rem = df_norm(df_add(sh.target, df_neg(mc)));
            const float need = (rem.hi + rem.lo) / gw;
            kept = need >= static_cast<float>(gc) ? static_cast<int>(gc) : static_cast<int>(ceilf(need));
          }
          if (kept < 1) kept = 1;
          if (kept > static_cast<int>(gc)) kept = static_cast<int>(gc);
          sh.vstar = gv;
          sh.gcount = (sh.phase == 1 && sh.floor_key != 0 && gkey == sh.floor_key) ? sh.k_gcount : static_cast<int>(gc);
          sh.gkept = kept;
          sh.zkept = df_norm(df_add(mc, df_mulf(df_make(gw), static_cast<float>(kept))));
          if (sh.phase == 0 && top_p < 1.f) {  // top-p on the renormalised top-k set, from the top again
            sh.k_vstar = sh.vstar;
            sh.k_gcount = sh.gcount;
            sh.k_gkept = kept;
            sh.zk = sh.zkept;
            sh.target = df_mulf(sh.zk, top_p);
            sh.floor_key = gkey;
            sh.floor_avail = kept;
            sh.phase = 1;
            sh.top_key = key_of_value(sh.m);
            sh.cnt_before = 0;
            sh.mass_before = df_make(0.f);
            start_window();
          } else {
            sh.phase = 2;
          }
        } else {
          // not in this window (cc, mc now hold its totals): go on below, or keep the whole set
          float below = -INFINITY;
          for (int w = 0; w < kWarps; ++w) below = fmaxf(below, sh.wf[w][2]);
          sh.cnt_before = cc;
          sh.mass_before = df_norm(mc);
          const bool floor_reached = sh.floor_key != 0 && sh.base_key <= sh.floor_key;
          if (sh.src_cands && (sh.base_key <= sh.line_key || !(below > -INFINITY))) {
            // the cut lies below what the list holds: search the rows from the top
            sh.src_cands = 0;
            reset_search();
          } else if (below > -INFINITY && !floor_reached) {
            sh.top_key = key_of_value(below);
            start_window();
          } else if (sh.phase == 0 && top_p < 1.f) {  // top-k keeps every token: top-p on the whole row
            sh.phase = 1;
            sh.floor_key = 0;
            sh.top_key = key_of_value(sh.m);
            sh.cnt_before = 0;
            sh.mass_before = df_make(0.f);
            start_window();
          } else {
            if (sh.floor_key != 0) {  // top-p keeps the whole top-k set
              sh.vstar = sh.k_vstar;
              sh.gcount = sh.k_gcount;
              sh.gkept = sh.k_gkept;
              sh.zkept = sh.zk;
            } else {
              sh.vstar = -INFINITY;
              sh.gcount = sh.gkept = 0;
              sh.zkept = sh.z;
            }
            sh.phase = 2;
          }
        }
      }
      __syncthreads();
    }
    if (tid == 0 && sh.phase != 2 && !sh.bad) {  // (not reached: at most 32 windows per phase)
      sh.vstar = -INFINITY;
      sh.gcount = sh.gkept = 0;
      sh.zkept = sh.z;
    }
    __syncthreads();
    // pass 3: the index of the last kept token of the cut group (lowest indices first)
    if (!sh.bad && sh.gkept > 0 && sh.gkept < sh.gcount && sh.src_cands) {
      // from the list: the tokens of the cut value, sorted by index (the list is unordered)
      const float vs = sh.vstar;
      if (tid == 0) sh.tie_seen = 0;
      __syncthreads();
      for (int e = tid; e < kCap; e += kThreads) {
        if ((e & (kSegCap - 1)) >= sh.wcnt[e / kSegCap]) continue;
        const uint2 en = mylist[e];
        if (Elt<DT>::value(en.y) == vs) hist[atomicAdd(&sh.tie_seen, 1u)] = en.x - 1u;
      }
      __syncthreads();
      const int g = static_cast<int>(sh.tie_seen);
      int np2 = 1;
      while (np2 < g) np2 <<= 1;
      for (int e = g + tid; e < np2; e += kThreads) hist[e] = 0xFFFFFFFFu;
      __syncthreads();
      bitonic_sort(hist, np2);
      if (tid == 0) sh.tie_last = static_cast<int>(hist[sh.gkept - 1]);
      __syncthreads();
    } else if (!sh.bad && sh.gkept > 0 && sh.gkept < sh.gcount) {
      const float vs = sh.vstar;
      if (tid == 0) {
        sh.tie_target = sh.gkept;
        sh.tie_seen = 0;
        sh.tie_found = -1;
      }
      __syncthreads();
      ok = stream_rows<DT>(sh, ring, rows1, 1, V, aligned, 0, nchunks, [&](int ch, uint32_t st, int nvec) {
        if (sh.tie_found >= 0) return;  // (uniform: read after the stream's barrier)
        uint32_t cv[kVPT];
        uint32_t tot = 0;
#pragma unroll
        for (int j = 0; j < kVPT; ++j) {
          const int v = tid + j * kThreads;
          uint32_t n = 0;
          if (v < nvec) {
            const uint4 q = lds128(st + 16u * v);
#pragma unroll
            for (int jj = 0; jj < PV; ++jj) n += val<DT>(q, jj) == vs;
          }
          cv[j] = n;
          tot += n;
        }
        tot = __reduce_add_sync(kFullMask, tot);
        if (lane == 0) sh.wu[warp][1] = tot;
        __syncthreads();
        uint32_t all = 0;
        for (int w = 0; w < kWarps; ++w) all += sh.wu[w][1];
        const uint32_t seen = sh.tie_seen;
        const uint32_t want = static_cast<uint32_t>(sh.tie_target);
        __syncthreads();
        if (seen + all < want) {
          if (tid == 0) sh.tie_seen = seen + all;
          return;
        }
        // the chunk holds it: rounds of kThreads vectors in index order
        uint32_t base_seen = seen;
        for (int j = 0; j < kVPT; ++j) {
          uint32_t incl = cv[j];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
            if (lane >= o) incl += y;
          }
          if (lane == 31) sh.wu[warp][0] = incl;
          __syncthreads();
          uint32_t pre = 0, rt = 0;
          for (int w = 0; w < kWarps; ++w) {
            if (w < warp) pre += sh.wu[w][0];
            rt += sh.wu[w][0];
          }
          incl += pre;
          const uint32_t before = base_seen + incl - cv[j];
          if (cv[j] > 0 && before < want && base_seen + incl >= want) {
            const int v = tid + j * kThreads;
            const uint4 q = lds128(st + 16u * v);
            uint32_t left = want - before;
            int jj = 0;
            for (; jj < PV; ++jj)
              if (val<DT>(q, jj) == vs && --left == 0) break;
            sh.tie_found = ch * epc + v * PV + jj;
            sh.stop = 1;
          }
          __syncthreads();
          base_seen += rt;
          if (sh.tie_found >= 0) break;
        }
      });
      if (tid == 0) sh.tie_last = sh.tie_found >= 0 ? sh.tie_found : 0x7FFFFFFF;
      __syncthreads();
    }
  }


  // a draft row's list serves only its own cut: back to zero now
  if (FILTER && !is_target)
    for (int e = tid; e < kCap; e += kThreads)
      if ((e & (kSegCap - 1)) < sh.wcnt[e / kSegCap]) mylist[e] = make_uint2(0u, 0u);
  // ---- the row's probability at the draft token; publish; the pair's accept test
  if (tid == 0) {
    const float zk = sh.zkept.hi + sh.zkept.lo;
    const float izk = (!sh.bad && zk > 0.f) ? 1.f / zk : 0.f;
    float xp = 0.f;
    if (i < k && x >= 0 && x < V && !sh.bad) {
      const bool kept = xv > sh.vstar || (xv == sh.vstar && x <= sh.tie_last);
      xp = kept ? mass(xv, sh.c, sh.nmc) * izk : 0.f;
    }
    RowOut o;
    o.m = sh.m;
    o.c = sh.c;
    o.nmc = sh.nmc;
    o.bad = sh.bad;
    o.zh = sh.z.hi;
    o.zl = sh.z.lo;
    o.vstar = sh.vstar;
    o.tie_last = sh.tie_last;
    o.kh = sh.zkept.hi;
    o.kl = sh.zkept.lo;
    o.izk = izk;
    o.xprob = xp;
    o.accept = 0;
    o.ncand = sh.overflow ? -1 : sh.ncand;
    o.cands_ok = FILTER && !sh.bad && sh.src_cands;  // the kept set was found within the list
    o.nwritten = 0;
    *me = o;
    if (sh.bad) atomicOr(a.status, sh.timed_out ? SPEC_STATUS_TIMEOUT | SPEC_STATUS_BAD_ROW : SPEC_STATUS_BAD_ROW);
    __threadfence();
    sh.assemble = 0;  // here: this CTA posts a sequence event
    sh.dodraw = 0;
    sh.drawn = -2;    // -2: this position writes no token
    if (i < k) {
      const uint32_t old = atomicAdd(a.done + static_cast<size_t>(b) * k + i, 1u);
      if (old == 1u) {  // the second row of the pair: the accept test
        __threadfence();
        const RowOut* pt = outs + static_cast<size_t>(b) * R + 2 * i;
        for (int q = 0; q < 2; ++q)
          for (int f = 0; f < static_cast<int>(sizeof(RowOut) / 4); ++f)
            reinterpret_cast<uint32_t*>(&sh.ro[q])[f] = __ldcg(reinterpret_cast<const uint32_t*>(pt + q) + f);
        const int bad = sh.ro[0].bad | sh.ro[1].bad;
        const float px = sh.ro[0].xprob, qx = sh.ro[1].xprob;
        const float u = a.uniforms[static_cast<size_t>(b) * (k + 2) + i];
        const bool in_range = x >= 0 && x < V;
        const bool acc = !bad && in_range && u * qx < px;
        if (a.out_p) a.out_p[static_cast<size_t>(b) * k + i] = bad ? 0.f : px;
        if (a.out_q) a.out_q[static_cast<size_t>(b) * k + i] = bad ? 0.f : qx;
        if (!in_range) atomicOr(a.status, SPEC_STATUS_BAD_TOKEN);
        if (!acc) {
          // draw here unless an earlier position of the sequence is known to have rejected
          const uint32_t rc = *rej_word;
          atomicMax(a.draw_tickets + b, static_cast<uint32_t>(k + 1 - i));
          sh.dodraw = !bad && !(rc > static_cast<uint32_t>(k + 1 - i));
          sh.drawn = -1;
        }
        sh.assemble = 1;
      }
    } else {  // the bonus row: draws unless a rejection is known
      sh.ro[0] = o;
      sh.dodraw = !sh.bad && *rej_word == 0u;
      sh.drawn = -1;
      sh.assemble = 1;
    }
  }
  __syncthreads();
  if (sh.dodraw) {
    const bool pair = i < k;
    const unsigned char* tr = trow_base + (static_cast<size_t>(b) * (k + 1) + i) * V * E;
    const unsigned char* dr = pair ? drow_base + (static_cast<size_t>(b) * k + i) * V * E : nullptr;
    const bool dal = a.aligned_target && (!pair || a.aligned_draft);
    const float u = a.uniforms[static_cast<size_t>(b) * (k + 2) + (pair ? k + 1 : k)];
    int t;
    if (FILTER && sh.ro[0].cands_ok) {  // the target's kept set is listed: draw over it, sorted by index
      const uint2* tl = lists + (static_cast<size_t>(b) * R + 2 * i) * kCap;
      unsigned long long* srt = reinterpret_cast<unsigned long long*>(hist);
      const float vsp = sh.ro[0].vstar;
      const int tlp = sh.ro[0].tie_last;
      if (tid == 0) sh.tie_seen = 0;
      __syncthreads();
      for (int e = tid; e < kCap; e += kThreads) {
        const uint2 en = __ldcg(tl + e);
        if (en.x == 0u) continue;
        const float lp = Elt<DT>::value(en.y);
        const uint32_t idx = en.x - 1u;
        if (lp > vsp || (lp == vsp && static_cast<int>(idx) <= tlp))
          srt[atomicAdd(&sh.tie_seen, 1u)] = (static_cast<unsigned long long>(idx) << 32) | en.y;
      }
      __syncthreads();
      const int nk = static_cast<int>(sh.tie_seen);
      int np2 = 1;
      while (np2 < nk) np2 <<= 1;
      for (int e = nk + tid; e < np2; e += kThreads) srt[e] = ~0ull;
      __syncthreads();
      bitonic_sort(srt, np2);
      t = draw_cands<DT>(sh, ctot, srt, nk, dr, u);
    } else {
      t = draw_token<DT>(sh, ring, ctot, tr, dr, V, dal, u);
    }
    if (tid == 0) sh.drawn = t;
    __syncthreads();
  }
  // the target row's list has served its last use (the pair's accept test and draw, or the bonus draw)
  if (FILTER && sh.assemble) {
    uint2* tl = lists + (static_cast<size_t>(b) * R + 2 * i) * kCap;
    for (int e = tid; e < kCap; e += kThreads)
      if (__ldcg(&tl[e].x) != 0u) tl[e] = make_uint2(0u, 0u);
  }
  // ---- the sequence: the last event writes the committed tokens and clears the counters
  if (tid == 0 && sh.assemble) {
    int32_t* otok = a.out_tokens + static_cast<size_t>(b) * (k + 1);
    if (sh.drawn != -2) otok[i] = sh.drawn;
    __threadfence();
    const uint32_t old = atomicAdd(a.seq_tickets + b, 1u);
    sh.assemble = 0;
    if (old == static_cast<uint32_t>(k)) {
      __threadfence();
      const uint32_t rc = *rej_word;
      // (a rejection word outside 1..k+1 cannot come from this kernel; n stays in range regardless)
      const int n = (rc >= 1u && rc <= static_cast<uint32_t>(k + 1)) ? k + 1 - static_cast<int>(rc) : k;
      const int32_t tn = __ldcg(otok + n);
      const int32_t* tok = a.tokens + static_cast<size_t>(b) * k;
      for (int j = 0; j < n; ++j) otok[j] = tok[j];
      otok[n] = tn;
      for (int j = n + 1; j <= k; ++j) otok[j] = -1;
      a.out_n[b] = n;
      for (int j = 0; j < k; ++j) a.done[static_cast<size_t>(b) * k + j] = 0u;
      a.seq_tickets[b] = 0u;
      a.draw_tickets[b] = 0u;
      sh.assemble = 1;
    }
  }
  __syncthreads();
  if (sh.assemble) {  // the sequence's row records go back to zero (the workspace is zero between calls)
    uint32_t* rec = reinterpret_cast<uint32_t*>(outs + static_cast<size_t>(b) * R);
    for (int w = tid; w < R * static_cast<int>(sizeof(RowOut) / 4); w += kThreads) rec[w] = 0u;
  }
  drain_ring(sh);
}

namespace {

constexpr int kRowMaxDevices = 64;
std::mutex g_row_mu;
bool g_row_ready[kRowMaxDevices][2][2];  // dynamic shared memory opted in, per device and kernel

template <int DT, bool FILTER>
int launch_row_t(const SampleArgs& a, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kRowMaxDevices) return cudaErrorInvalidDevice;
  auto kern = row_kernel<DT, FILTER>;
  const int smem = kStages * static_cast<int>(kStageBytes);
  {
    std::lock_guard<std::mutex> lock(g_row_mu);
    if (!g_row_ready[dev][DT][FILTER ? 1 : 0]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      g_row_ready[dev][DT][FILTER ? 1 : 0] = true;
    }
  }
  const unsigned grid = static_cast<unsigned>(a.B) * static_cast<unsigned>(2 * a.k + 1);
  kern<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool row_supported(const SampleArgs& a, int dtype) {
  const bool filter = a.top_k > 0 || a.top_p < 1.f;
  if (a.mode != MODE_SAMPLE || a.k < 1) return false;
  if (filter && dtype != DT_BF16) return false;
  // the draw keeps per-warp totals for every chunk of two rows
  const size_t e = dtype == DT_BF16 ? 2 : 4;
  const size_t chunks = (static_cast<size_t>(a.V) * e + kStageBytes / 2 - 1) / (kStageBytes / 2);
  return chunks <= static_cast<size_t>(kMaxChunks);
}

int launch_rows(const SampleArgs& a, int dtype, void* stream) {
  const bool filter = a.top_k > 0 || a.top_p < 1.f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == DT_BF16) return filter ? launch_row_t<DT_BF16, true>(a, st) : launch_row_t<DT_BF16, false>(a, st);
  return launch_row_t<DT_F32, false>(a, st);
}

}  // namespace specv
