// tree_sample_kernel.cu -- token-tree sampling verification.
//
// The accept-or-correct rule of speculative sampling (Edge Inference Notes,
// post on speculative decoding and EAGLE-3, "The core idea: draft, then
// check", step 3) applied down the branches of a draft tree ("One decode
// round, end to end").  At a node v with target distribution p and draft
// distribution q (temperature T), the children are tried in ascending node
// order: child x is accepted iff u_x q(x) < r(x), where r starts as p and,
// after each rejected child, becomes max(0, r - q) renormalised.  With
// c_0 = 0, W_0 = 1 that residual is  r_m = max(0, p - c_m q) / W_m  with
// c_{m+1} = c_m + W_m and W_{m+1} = sum_t max(0, p_t - c_{m+1} q_t); a mass of
// zero puts r back to p.  When no child is accepted one token is drawn from r
// (inverse CDF in ascending index order, uniform u_0).
//
// Which children a node accepts depends only on that node's rows, its
// children's tokens and their uniforms, never on how the walk reached the
// node.  So every node with children to test is decided independently and in
// parallel (tree_node_kernel): one thread-block cluster of kTreeCl CTAs per
// node copies the node's target and draft rows into shared memory (bulk
// copies, CTA r a 1/kTreeCl slice of each), reduces the row maxima and masses
// through distributed shared memory, then runs the sibling loop, one
// residual-mass pass over the shared-memory slices per rejected child.  A
// node that accepts no child records its stop residual's per-chunk sums.
// Nodes without children to test are only marked: their stop distribution
// is p itself.  tree_walk_kernel (one cluster per tree) then follows the
// accepted children from the root; if the walk stops at a marked node, the
// cluster computes that node's p chunk sums, and the correction is drawn:
// the chunk from the sums, the element within it from the rows.
//
// Masses are 2^(l c + nm) with c = log2(e)/T and nm = -max * c, one ex2 per
// element.  Sums are float per lane and double-float (an unevaluated sum of
// two floats) across lanes, warps and CTAs: this GPU's fp64 pipe is narrow,
// and every fp64 instruction on a reduction or a decision sits on a chain
// that one thread waits for.  They are always taken in the same order, so
// every CTA of a cluster takes the same decisions; the accept test and the
// draw compare double-float values.

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <math.h>
#include <stdint.h>

#include "device_common.cuh"
#include "internal.h"

namespace specv {

namespace {

constexpr uint32_t kPiece = 16384;  // bytes per bulk copy
constexpr int kPre = 32;            // children whose logits are fetched ahead of the sibling loop
constexpr int16_t kNoParent = -2;   // a parent entry outside [-1, N)

// ------------------------------------------------ double-float arithmetic
// A value hi + lo with |lo| at most half an ulp of hi: TwoSum for additions,
// an fma for the rounding error of a product.
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF df_norm(DF a) {  // Fast2Sum
  const float s = a.hi + a.lo;
  return DF{s, a.lo - (s - a.hi)};
}
__device__ __forceinline__ DF df_two(float x, float y) {  // x + y exactly
  const float s = x + y;
  const float bp = s - x;
  return DF{s, (x - (s - bp)) + (y - bp)};
}
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const DF s = df_two(a.hi, b.hi);
  return df_norm(DF{s.hi, s.lo + (a.lo + b.lo)});
}
__device__ __forceinline__ DF df_sub(DF a, DF b) { return df_add(a, DF{-b.hi, -b.lo}); }
__device__ __forceinline__ DF df_mulf(DF a, float f) {
  const float p = a.hi * f;
  return df_norm(DF{p, fmaf(a.lo, f, fmaf(a.hi, f, -p))});
}
__device__ __forceinline__ DF df_mul(DF a, DF b) {
  const float p = a.hi * b.hi;
  return df_norm(DF{p, fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, fmaf(a.hi, b.hi, -p)))});
}
__device__ __forceinline__ bool df_gt(DF a, DF b) { return df_sub(a, b).hi > 0.f; }
__device__ __forceinline__ bool df_pos(DF a) { return a.hi > 0.f; }  // of a normalised value
__device__ __forceinline__ float df_f(DF a) { return a.hi + a.lo; }
__device__ __forceinline__ DF shfl_df(DF a, int src) {
  return DF{__shfl_sync(0xFFFFFFFFu, a.hi, src), __shfl_sync(0xFFFFFFFFu, a.lo, src)};
}
__device__ __forceinline__ DF shfl_up_df(DF a, int d) {
  return DF{__shfl_up_sync(0xFFFFFFFFu, a.hi, d), __shfl_up_sync(0xFFFFFFFFu, a.lo, d)};
}
__device__ __forceinline__ DF shfl_down_df(DF a, int d) {
  return DF{__shfl_down_sync(0xFFFFFFFFu, a.hi, d), __shfl_down_sync(0xFFFFFFFFu, a.lo, d)};
}
// Sum over the warp, valid in lane 0.
__device__ __forceinline__ DF warp_sum_df(DF v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = df_add(v, shfl_down_df(v, o));
  return v;
}

struct TreeShm {
  uint64_t bar[2];           // bulk-copy completion: target slice, draft slice
  float red[2][8];           // per-CTA values handed to the cluster, by round parity
  float gm[2];               // cluster-wide maxima (target, draft)
  DF gz[2];                  // cluster-wide masses relative to them
  DF gsum;                   // cluster-wide sum of the last residual pass
  int gbad;                  // a slice of the cluster holds NaN / +inf (or did not arrive)
  DF wsum[kWarps][2];        // per-warp sums of the current pass
  DF zc[kWarps];             // per-warp sums of 2^(l c + nmp) (the c = 0 residual)
  DF wc[kWarps];             // per-warp sums of the last residual pass
  float fmax[kWarps][2];
  int bad[kWarps];
  int16_t kids[kMaxTreeNodes];
  int16_t par[kMaxTreeNodes];
  int nk_w[kWarps];
  float kl[kPre], kd[kPre], ku[kPre];  // the first children's target / draft logits and uniforms
  float mloc[2];             // this CTA's maxima (target, draft)
  int badloc;               // this CTA's slices hold NaN / +inf (or did not arrive)
  int nk, has_child, accept, timed_out;
  int next[2];               // rank 0: the next work item claimed, by node parity
  int nextl;                 // that item, read by every CTA of the cluster
  int walk_v, walk_n, walk_ok, draw_w, draw_past;
  DF draw_rem;
};

template <int DT>
__device__ __forceinline__ bool bad_bits(uint32_t b) {
  // NaN or +inf; -inf is an ordinary masked logit
  if (DT == DT_BF16) return (b & 0x7F80u) == 0x7F80u && b != 0xFF80u;
  return (b & 0x7F800000u) == 0x7F800000u && b != 0xFF800000u;
}

template <int DT>
__device__ __forceinline__ float smem_val(uint32_t base, int i) {
  if (DT == DT_BF16) return Elt<DT_BF16>::value(lds_u16(base + 2u * static_cast<uint32_t>(i)));
  return __uint_as_float(lds_u32(base + 4u * static_cast<uint32_t>(i)));
}

// The residual weight of one element; the c = 0 residual (fb == 0) is the
// target mass itself.  Used unchanged by the per-node passes and the draw.
__device__ __forceinline__ float resid_weight(float l, float d, float c, float nmp, float nmq, float fa,
                                              float fb) {
  const float ep = ex2_approx(fmaf(l, c, nmp));
  if (fb == 0.f) return ep;
  const float eq = ex2_approx(fmaf(d, c, nmq));
  return fmaxf(0.f, fmaf(ep, fa, eq * -fb));
}

// ------------------------------------------------ packed float pairs (f32x2)
using u64 = unsigned long long;
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
// Masses 2^(l c + nm) of two elements: per half the same fma and ex2 as the
// scalar form in resid_weight.
__device__ __forceinline__ u64 mass2(u64 l2, u64 c2, u64 nm2) {
  float x, y;
  upk(fma2(l2, c2, nm2), x, y);
  return pkf(ex2_approx(x), ex2_approx(y));
}
// Residual weights of two elements: per half resid_weight with fb != 0.
__device__ __forceinline__ u64 resid2(u64 lp2, u64 lq2, u64 c2, u64 np2, u64 nq2, u64 fa2, u64 nfb2) {
  float x, y;
  upk(fma2(mass2(lp2, c2, np2), fa2, mul2(mass2(lq2, c2, nq2), nfb2)), x, y);
  return pkf(fmaxf(0.f, x), fmaxf(0.f, y));
}
// The element pairs of one 16-byte vector as float pairs.
template <int DT>
__device__ __forceinline__ u64 pair_of(const uint4& v, int h);
template <>
__device__ __forceinline__ u64 pair_of<DT_BF16>(const uint4& v, int h) {
  const uint32_t w = h == 0 ? v.x : h == 1 ? v.y : h == 2 ? v.z : v.w;
  return pk2(w << 16, w & 0xFFFF0000u);
}
template <>
__device__ __forceinline__ u64 pair_of<DT_F32>(const uint4& v, int h) {
  return h == 0 ? pk2(v.x, v.y) : pk2(v.z, v.w);
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Running maximum of a slice's 16-byte vectors, and whether it holds NaN or
// +inf.  bf16: four packed accumulators whose maximum propagates NaN, so one
// check at the end finds a bad value; f32: per element.
template <int DT>
struct VecMax;
template <>
struct VecMax<DT_BF16> {
  __nv_bfloat162 m[4];
  __device__ static __forceinline__ __nv_bfloat162 b2(uint32_t w) {
    __nv_bfloat162 r;
    *reinterpret_cast<uint32_t*>(&r) = w;
    return r;
  }
  __device__ __forceinline__ VecMax() {
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = b2(0xFF80FF80u);
  }
  __device__ __forceinline__ void add(const uint4& v) {
    m[0] = __hmax2_nan(m[0], b2(v.x));
    m[1] = __hmax2_nan(m[1], b2(v.y));
    m[2] = __hmax2_nan(m[2], b2(v.z));
    m[3] = __hmax2_nan(m[3], b2(v.w));
  }
  __device__ __forceinline__ void finish(float& mx, int& bad) const {
    const __nv_bfloat162 t = __hmax2_nan(__hmax2_nan(m[0], m[1]), __hmax2_nan(m[2], m[3]));
    const float r = max_nan(__low2float(t), __high2float(t));
    if (r != r || r == INFINITY) bad = 1;
    else mx = fmaxf(mx, r);
  }
};
template <>
struct VecMax<DT_F32> {
  float mx = -INFINITY;
  int bad = 0;
  __device__ __forceinline__ void add(const uint4& v) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t bits = Elt<DT_F32>::bits_of(v, e);
      bad |= bad_bits<DT_F32>(bits);
      mx = fmaxf(mx, __uint_as_float(bits));
    }
  }
  __device__ __forceinline__ void finish(float& m_out, int& bad_out) const {
    bad_out |= bad;
    m_out = fmaxf(m_out, mx);
  }
};

// log2(e) / T of tree b: the scalar temperature's factor, or the tree's own
// (the same float division as on the host).
__device__ __forceinline__ float tree_c(const TreeSampleArgs& a, int b) {
  return a.temps ? kLog2e / a.temps[b] : a.c;
}

__device__ __forceinline__ float warp_max_f32(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Warp 0, after a cluster barrier: lane l reads the first nv values that rank
// l % kTreeCl left in sh.red[slot] (one round of distributed-shared-memory
// reads, all lanes at once).
template <int NV>
__device__ __forceinline__ void cluster_read(TreeShm& sh, int slot, float (&v)[NV]) {
  const uint32_t base = mapa_shared(smem_addr(&sh.red[slot][0]), static_cast<int>(threadIdx.x) & (kTreeCl - 1));
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = ld_cluster_f32(base + 4u * i);
}

// The sum of one double-float per rank (lane r holds rank r's), in rank
// order.  Every lane adds the same shuffled values in the same order, so
// every lane, and every CTA of the cluster, holds the same bits.
__device__ __forceinline__ DF rank_sum(DF x) {
  DF s = shfl_df(x, 0);
#pragma unroll
  for (int r = 1; r < kTreeCl; ++r) s = df_add(s, shfl_df(x, r));
  return s;
}

// The maximum over ranks (lanes that differ in their low bits).
__device__ __forceinline__ float rank_max(float x) {
#pragma unroll
  for (int o = 1; o < kTreeCl; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
  return x;
}

// The cluster-wide sum of the double-float thread 0 of every CTA left in
// sh.red[slot][0..1], into sh.gsum.
__device__ void cluster_sum(TreeShm& sh, int slot) {
  cg::this_cluster().sync();
  if (threadIdx.x < 32) {
    float v[2];
    cluster_read(sh, slot, v);
    const DF s = rank_sum(DF{v[0], v[1]});
    if (threadIdx.x == 0) sh.gsum = s;
  }
  __syncthreads();
}

// Row statistics from per-CTA ones: sh.red[slot] = {max p, mass p (hi, lo),
// max q, mass q (hi, lo), bad} with masses relative to the CTA's own maxima.
// Into sh.gm / sh.gz / sh.gbad: the cluster maxima, and the masses relative
// to them (each CTA's mass scaled by 2^((m_r - m) c), summed in rank order).
__device__ void cluster_combine_stats(TreeShm& sh, int slot, float c) {
  cg::this_cluster().sync();
  if (threadIdx.x < 32) {
    float v[7];
    cluster_read(sh, slot, v);
    const float mp = rank_max(v[0]), mq = rank_max(v[3]), bad = rank_max(v[6]);
    // a CTA without mass (an empty or all -inf slice) adds nothing, and no 0 * NaN
    const DF zp = v[1] > 0.f ? df_mulf(DF{v[1], v[2]}, ex2_approx((v[0] - mp) * c)) : DF{0.f, 0.f};
    const DF zq = v[4] > 0.f ? df_mulf(DF{v[4], v[5]}, ex2_approx((v[3] - mq) * c)) : DF{0.f, 0.f};
    const DF sp = rank_sum(zp), sq = rank_sum(zq);
    if (threadIdx.x == 0) {
      sh.gm[0] = mp;
      sh.gm[1] = mq;
      sh.gz[0] = sp;
      sh.gz[1] = sq;
      sh.gbad = bad != 0.f;
    }
  }
  __syncthreads();
}

// Children of node j that are tested, in ascending node order, into sh.kids
// (sh.nk of them); sh.has_child tells whether j has any child at all.
__device__ void collect_children(const TreeSampleArgs& a, TreeShm& sh, const int32_t* tok, int j, bool testable) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int nk = 0, any = 0;
  for (int base = j + 1; base < a.N; base += kThreads) {
    const int jj = base + static_cast<int>(threadIdx.x);
    const bool child = jj < a.N && sh.par[jj] == j;
    const bool ok = child && testable && tok[jj] >= 0 && tok[jj] < a.V;
    any |= __syncthreads_or(child);
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, ok);
    if (lane == 0) sh.nk_w[warp] = __popc(bal);
    __syncthreads();
    int before = nk, total = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) before += sh.nk_w[w];
      total += sh.nk_w[w];
    }
    if (ok) sh.kids[before + __popc(bal & ((1u << lane) - 1u))] = static_cast<int16_t>(jj);
    nk += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    sh.nk = nk;
    sh.has_child = any;
  }
  __syncthreads();
}

// Thread 0: `bytes` from global src to shared dst by bulk copies completing on bar.
__device__ __forceinline__ void bulk_issue(uint64_t* bar, uint32_t dst, const unsigned char* src, uint32_t bytes) {
  mbar_arrive_expect_tx(bar, bytes);
  for (uint32_t off = 0; off < bytes; off += kPiece)
    bulk_copy_g2s_addr(dst + off, src + off, bytes - off < kPiece ? bytes - off : kPiece, bar);
}

// Thread 0: starts the bulk copies of this CTA's slices (16-byte aligned rows).
__device__ __forceinline__ void stage_issue(TreeShm& sh, const unsigned char* prow, const unsigned char* qrow,
                                            uint32_t bytes, bool with_q, uint32_t sp, uint32_t sq) {
  if (sh.timed_out) return;
  fence_proxy_async_smem();  // earlier reads of these slices come before the copies' writes
  bulk_issue(&sh.bar[0], sp, prow, bytes);
  if (with_q) bulk_issue(&sh.bar[1], sq, qrow, bytes);
}

// Brings elements [lo, lo+len) of the target row (and of the draft row when
// with_q) into shared memory -- bulk copies for 16-byte aligned rows (started
// here unless `issued`), plain loads otherwise -- and leaves this CTA's maxima
// in sh.mloc and its bad-value flag in sh.badloc.  A copy that does not
// complete within the bounded wait marks the slice bad and sets
// SPEC_STATUS_TIMEOUT; that CTA copies nothing more.
template <int DT>
__device__ void stage_rows(const TreeSampleArgs& a, TreeShm& sh, const unsigned char* prow,
                           const unsigned char* qrow, int len, bool with_q, uint32_t sp, uint32_t sq,
                           uint32_t& php, uint32_t& phq, bool issued) {
  constexpr int E = Elt<DT>::kBytes;
  constexpr int PV = Elt<DT>::kPerVec;
  float mp = -INFINITY, mq = -INFINITY;
  int bp = 0, bq = 0, tmo = 0;
  if (a.aligned) {
    const bool skip = sh.timed_out != 0;
    if (threadIdx.x == 0 && !issued) stage_issue(sh, prow, qrow, static_cast<uint32_t>(len) * E, with_q, sp, sq);
    bool ok = !skip;
    if (ok) {
      ok = mbar_wait_bounded(&sh.bar[0], php);
      php ^= 1u;
      if (with_q) {
        ok = mbar_wait_bounded(&sh.bar[1], phq) && ok;
        phq ^= 1u;
      }
    }
    if (!ok) {
      tmo = 1;
    } else {
      const int nv = len / PV;  // aligned rows: len is a whole number of vectors
      VecMax<DT> xp, xq;
      for (int v = threadIdx.x; v < nv; v += kThreads) {
        xp.add(lds128(sp + 16u * v));
        if (with_q) xq.add(lds128(sq + 16u * v));
      }
      xp.finish(mp, bp);
      if (with_q) xq.finish(mq, bq);
    }
  } else {
    for (int i = threadIdx.x; i < len; i += kThreads) {
      const uint32_t b1 = Elt<DT>::bits_at(prow, i);
      bp |= bad_bits<DT>(b1);
      mp = fmaxf(mp, Elt<DT>::value(b1));
      if (E == 2) sts_u16(sp + 2u * i, b1); else sts_u32(sp + 4u * i, b1);
      if (with_q) {
        const uint32_t b2 = Elt<DT>::bits_at(qrow, i);
        bq |= bad_bits<DT>(b2);
        mq = fmaxf(mq, Elt<DT>::value(b2));
        if (E == 2) sts_u16(sq + 2u * i, b2); else sts_u32(sq + 4u * i, b2);
      }
    }
    // pad the last vector with -inf: the passes read whole vectors
    const int pad = (len + PV - 1) / PV * PV - len;
    if (static_cast<int>(threadIdx.x) < pad) {
      const int i = len + threadIdx.x;
      if (E == 2) {
        sts_u16(sp + 2u * i, 0xFF80u);
        if (with_q) sts_u16(sq + 2u * i, 0xFF80u);
      } else {
        sts_u32(sp + 4u * i, 0xFF800000u);
        if (with_q) sts_u32(sq + 4u * i, 0xFF800000u);
      }
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  mp = warp_max_f32(mp);
  mq = warp_max_f32(mq);
  bp = __any_sync(0xFFFFFFFFu, bp);
  bq = __any_sync(0xFFFFFFFFu, bq);
  tmo = __any_sync(0xFFFFFFFFu, tmo);
  if (lane == 0) {
    sh.fmax[warp][0] = mp;
    sh.fmax[warp][1] = mq;
    sh.bad[warp] = bp | (bq << 1) | (tmo << 2);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float m0 = -INFINITY, m1 = -INFINITY;
    int bd = 0;
    for (int w = 0; w < kWarps; ++w) {
      m0 = fmaxf(m0, sh.fmax[w][0]);
      m1 = fmaxf(m1, sh.fmax[w][1]);
      bd |= sh.bad[w];
    }
    if ((bd & 4) || (a.aligned && sh.timed_out)) {  // no data this time: the slice counts as bad
      if (!sh.timed_out) atomicOr(a.status, SPEC_STATUS_TIMEOUT);
      sh.timed_out = 1;
      bd |= 1;
    }
    sh.mloc[0] = m0;
    sh.mloc[1] = m1;
    sh.badloc = (bd & 1) | (with_q ? (bd >> 1) & 1 : 0);
  }
  __syncthreads();
}

// This CTA's masses relative to its own maxima (one pass), handed to the
// cluster with the maxima (the layout cluster_combine_stats reads); sh.zc
// keeps the per-warp target masses.  Then the cluster-wide statistics in
// sh.gm, sh.gz and sh.gbad.
template <int DT>
__device__ void slice_stats(TreeShm& sh, uint32_t sp, uint32_t sq, int len, int wchunk, bool with_q, float c,
                            int slot);

// Sums over this CTA's slice, per warp chunk: 16-byte vectors, lanes
// interleaved, float pairs per lane (two accumulators), double-float across
// lanes.
// The slice is whole vectors (lenv elements; an unaligned slice is padded
// with -inf, which has no mass and no weight).  MODE 0: target and draft
// masses (sh.wsum[w][0], [1]);  MODE 1: residual weights (sh.wsum[w][0]).
template <int DT, int MODE>
__device__ void slice_pass(TreeShm& sh, uint32_t sp, uint32_t sq, int lenv, int wchunk, bool with_q, float c,
                           float nmp, float nmq, float fa, float fb) {
  constexpr int PV = Elt<DT>::kPerVec;
  constexpr int NP = PV / 2;  // element pairs per vector
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wlo = warp * wchunk;
  const int whi = min(lenv, wlo + wchunk);
  const u64 c2 = pkf(c, c), np2 = pkf(nmp, nmp), nq2 = pkf(nmq, nmq), fa2 = pkf(fa, fa), nfb2 = pkf(-fb, -fb);
  u64 a0 = 0ull, a1 = 0ull, b0 = 0ull, b1 = 0ull;
  for (int i0 = wlo + lane * PV; i0 < whi; i0 += 32 * PV) {
    const uint32_t off = 16u * static_cast<uint32_t>(i0 / PV);
    const uint4 x = lds128(sp + off);
    if (MODE == 0) {
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        if (h & 1) a1 = add2(a1, mass2(pair_of<DT>(x, h), c2, np2));
        else a0 = add2(a0, mass2(pair_of<DT>(x, h), c2, np2));
      }
      if (with_q) {
        const uint4 y = lds128(sq + off);
#pragma unroll
        for (int h = 0; h < NP; ++h) {
          if (h & 1) b1 = add2(b1, mass2(pair_of<DT>(y, h), c2, nq2));
          else b0 = add2(b0, mass2(pair_of<DT>(y, h), c2, nq2));
        }
      }
    } else {
      const uint4 y = lds128(sq + off);
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        const u64 r2 = resid2(pair_of<DT>(x, h), pair_of<DT>(y, h), c2, np2, nq2, fa2, nfb2);
        if (h & 1) a1 = add2(a1, r2);
        else a0 = add2(a0, r2);
      }
    }
  }
  float x0, y0, x1, y1;
  upk(add2(a0, a1), x0, y0);
  upk(add2(b0, b1), x1, y1);
  const DF d0 = warp_sum_df(df_two(x0, y0));
  const DF d1 = MODE == 0 ? warp_sum_df(df_two(x1, y1)) : DF{0.f, 0.f};
  if (lane == 0) {
    sh.wsum[warp][0] = d0;
    sh.wsum[warp][1] = d1;
  }
  __syncthreads();
}


template <int DT>
__device__ void slice_stats(TreeShm& sh, uint32_t sp, uint32_t sq, int len, int wchunk, bool with_q, float c,
                            int slot) {
  const float m0 = sh.mloc[0], m1 = with_q ? sh.mloc[1] : -INFINITY;
  const float nm0 = m0 == -INFINITY ? 0.f : -m0 * c;  // an empty or all -inf slice has no mass
  const float nm1 = m1 == -INFINITY ? 0.f : -m1 * c;
  slice_pass<DT, 0>(sh, sp, sq, len, wchunk, with_q, c, nm0, nm1, 0.f, 0.f);
  if (threadIdx.x == 0) {
    DF z0 = sh.wsum[0][0], z1 = sh.wsum[0][1];
    sh.zc[0] = z0;
    for (int w = 1; w < kWarps; ++w) {
      sh.zc[w] = sh.wsum[w][0];
      z0 = df_add(z0, sh.wsum[w][0]);
      z1 = df_add(z1, sh.wsum[w][1]);
    }
    sh.red[slot][0] = m0;
    sh.red[slot][1] = z0.hi;
    sh.red[slot][2] = z0.lo;
    sh.red[slot][3] = m1;
    sh.red[slot][4] = z1.hi;
    sh.red[slot][5] = z1.lo;
    sh.red[slot][6] = static_cast<float>(sh.badloc);
  }
  cluster_combine_stats(sh, slot, c);
}

// Parents of tree b into sh.par (entries outside [-1, N) become kNoParent).
// The plan kernel has already checked that every listed node is attached
// below max_depth.
__device__ void stage_parents(const TreeSampleArgs& a, TreeShm& sh, int b) {
  const int32_t* par = a.parents + static_cast<size_t>(b) * a.N;
  for (int i = threadIdx.x; i < a.N; i += kThreads) {
    const int p = par[i];
    sh.par[i] = static_cast<int16_t>(p >= -1 && p < a.N ? p : kNoParent);
  }
  __syncthreads();
}

// The correction drawn at stop node v of tree b (n nodes accepted) by one
// CTA: the chunk by a double-float prefix over the node's chunk sums, then
// the warp sub-range and the element from the node's rows.  The chunk sums
// and the residual's parameters come from the node's record, or, for a stop
// node whose p the walk's cluster has just summed (`local`), from every
// CTA's sh.wc by distributed-shared-memory reads and from the arguments.
template <int DT>
__device__ void draw_at(const TreeSampleArgs& a, TreeShm& sh, int b, int v, int n, bool local, float nmp,
                        float nmq, float fa, float fb) {
  constexpr int E = Elt<DT>::kBytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int D = a.max_depth + 1;
  int32_t* otok = a.out_tokens + static_cast<size_t>(b) * D;
  const size_t g = static_cast<size_t>(b) * a.N + v;
  const TreeRec* r = a.recs + g;
  if (!local) {
    nmp = __ldcg(&r->nmp);
    nmq = __ldcg(&r->nmq);
    fa = __ldcg(&r->fa);
    fb = __ldcg(&r->fb);
  }
  const unsigned char* lrow = static_cast<const unsigned char*>(a.logits) + g * a.V * E;
  const unsigned char* drow = static_cast<const unsigned char*>(a.draft) + g * a.V * E;
  if (warp == 0) {
    // chunk: lane L holds chunks 2L and 2L+1 (chunk i is warp i % kWarps of rank i / kWarps)
    DF c0, c1;
    if (local) {
      const int rk = 2 * lane / kWarps, w0 = 2 * lane % kWarps;
      const uint32_t p0 = mapa_shared(smem_addr(&sh.wc[w0]), rk), p1 = mapa_shared(smem_addr(&sh.wc[w0 + 1]), rk);
      c0 = DF{ld_cluster_f32(p0), ld_cluster_f32(p0 + 4u)};
      c1 = DF{ld_cluster_f32(p1), ld_cluster_f32(p1 + 4u)};
    } else {
      c0 = DF{__ldcg(&r->chunk[2 * lane][0]), __ldcg(&r->chunk[2 * lane][1])};
      c1 = DF{__ldcg(&r->chunk[2 * lane + 1][0]), __ldcg(&r->chunk[2 * lane + 1][1])};
    }
    const DF own = df_add(c0, c1);
    DF incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const DF y = shfl_up_df(incl, o);
      if (lane >= o) incl = df_add(incl, y);
    }
    const DF total = shfl_df(incl, 31);
    const DF target = df_mulf(total, a.uniforms[static_cast<size_t>(b) * a.N]);
    const uint32_t over = __ballot_sync(0xFFFFFFFFu, df_gt(incl, target));
    const uint32_t pos = __ballot_sync(0xFFFFFFFFu, df_pos(c0) || df_pos(c1));
    int l = -1;
    if (over) l = __ffs(over) - 1;
    else if (pos) l = 31 - __clz(pos);
    int ci = -1;
    DF rem{0.f, 0.f};
    if (l >= 0) {
      const DF ex = shfl_df(df_sub(incl, own), l);
      const DF a0 = shfl_df(c0, l), a1 = shfl_df(c1, l);
      if (over) {
        ci = (df_gt(df_add(ex, a0), target) || !df_pos(a1)) ? 2 * l : 2 * l + 1;
      } else {
        ci = df_pos(a1) ? 2 * l + 1 : 2 * l;
      }
      rem = df_sub(target, ci & 1 ? df_add(ex, a0) : ex);
    }
    if (lane == 0) {
      sh.draw_w = ci;
      sh.draw_rem = rem;
    }
  }
  __syncthreads();
  const int ci = sh.draw_w;
  if (ci < 0) {  // no positive weight anywhere: nothing to draw from
    if (tid == 0) {
      otok[n] = -1;
      a.out_n[b] = n;
      atomicOr(a.status, SPEC_STATUS_BAD_ROW);
    }
    __syncthreads();
    return;
  }
  const int cr = ci / kWarps, cw = ci % kWarps;
  const int slo = cr * a.slice;
  const int slen = max(0, min(a.V, slo + a.slice) - slo);
  const int clo = slo + min(slen, cw * a.wchunk);
  const int chi = slo + min(slen, (cw + 1) * a.wchunk);
  const int sub = ((chi - clo + kWarps - 1) / kWarps + 31) / 32 * 32;
  {
    const int wlo = min(chi, clo + warp * sub), whi = min(chi, clo + (warp + 1) * sub);
    float s = 0.f;
#pragma unroll 8
    for (int t = wlo + lane; t < whi; t += 32)
      s += resid_weight(Elt<DT>::value(Elt<DT>::bits_at(lrow, t)),
                        fb == 0.f ? 0.f : Elt<DT>::value(Elt<DT>::bits_at(drow, t)), tree_c(a, b), nmp, nmq, fa, fb);
    const DF ws = warp_sum_df(DF{s, 0.f});
    if (lane == 0) sh.wsum[warp][0] = ws;
  }
  __syncthreads();
  if (tid == 0) {
    const DF rem = sh.draw_rem;
    DF cum{0.f, 0.f};
    int pick = -1, lastpos = -1;
    for (int w = 0; w < kWarps; ++w) {
      const DF s = sh.wsum[w][0];
      if (df_pos(s)) lastpos = w;
      if (df_pos(s) && df_gt(df_add(cum, s), rem)) {
        pick = w;
        break;
      }
      cum = df_add(cum, s);
    }
    sh.draw_past = pick < 0;  // past every element: the last positive one
    if (pick < 0) pick = lastpos;
    else sh.draw_rem = df_sub(rem, cum);
    sh.walk_v = pick;
  }
  __syncthreads();
  const int pick = sh.walk_v;
  if (warp == (pick < 0 ? 0 : pick)) {
    int token = -1;
    if (pick >= 0) {
      const DF rem = sh.draw_rem;
      const bool past = sh.draw_past != 0;
      const int wlo = min(chi, clo + pick * sub), whi = min(chi, clo + (pick + 1) * sub);
      DF acc{0.f, 0.f};
      constexpr int kAhead = 8;  // rounds of 32 elements fetched before they are scanned
      bool found = false;
      for (int base0 = wlo; base0 < whi && !found; base0 += 32 * kAhead) {
        float w[kAhead];
#pragma unroll
        for (int k = 0; k < kAhead; ++k) {
          const int t = base0 + 32 * k + lane;
          w[k] = t < whi ? resid_weight(Elt<DT>::value(Elt<DT>::bits_at(lrow, t)),
                                        fb == 0.f ? 0.f : Elt<DT>::value(Elt<DT>::bits_at(drow, t)), tree_c(a, b), nmp,
                                        nmq, fa, fb)
                         : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kAhead; ++k) {
          const int base = base0 + 32 * k;
          // 32 weights: a float prefix, added to the double-float sum before them
          const float incl = warp_incl_scan(w[k]);
          const uint32_t hit = __ballot_sync(0xFFFFFFFFu, w[k] > 0.f && !past && df_gt(df_add(acc, DF{incl, 0.f}), rem));
          const uint32_t pos = __ballot_sync(0xFFFFFFFFu, w[k] > 0.f);
          if (!found) {
            if (pos) token = base + 31 - __clz(pos);
            if (hit) {
              token = base + __ffs(hit) - 1;
              found = true;
            }
          }
          acc = df_add(acc, DF{__shfl_sync(0xFFFFFFFFu, incl, 31), 0.f});
        }
      }
    }
    if (lane == 0) {
      otok[n] = token;
      a.out_n[b] = n;
      if (token < 0) atomicOr(a.status, SPEC_STATUS_BAD_ROW);
    }
  }
  __syncthreads();
}


// One CTA per tree: validates the parents, finds every node's depth, and
// lists the nodes with at least one child to test (attached, above
// max_depth, a child whose token is in [0, V)) for tree_node_kernel; the
// others get their final record here (detached, or stop residual p).
__global__ void __launch_bounds__(kThreads) tree_plan_kernel(const TreeSampleArgs a) {
  __shared__ int16_t par[kMaxTreeNodes];
  __shared__ int16_t dep[kMaxTreeNodes];
  __shared__ uint8_t has_child[kMaxTreeNodes];
  __shared__ int testable_child[kMaxTreeNodes];  // children to test, per node
  __shared__ int16_t raw[kMaxTreeNodes];
  __shared__ int16_t list[kMaxTreeNodes];
  __shared__ int order_key[kMaxTreeNodes];
  __shared__ int cnt, base;
  const int b = blockIdx.x, tid = threadIdx.x, N = a.N;
  // a tree temperature that gives no distribution: every node bad, nothing listed
  const bool bad_t = a.temps != nullptr && !(a.temps[b] > 0.f && isfinite(a.temps[b]));
  const int32_t* pg = a.parents + static_cast<size_t>(b) * N;
  const int32_t* tok = a.tokens + static_cast<size_t>(b) * N;
  uint32_t st = 0;
  for (int i = tid; i < N; i += kThreads) {
    const int p = pg[i];
    par[i] = static_cast<int16_t>(p >= -1 && p < N ? p : kNoParent);
    has_child[i] = 0;
    testable_child[i] = 0;
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) st |= SPEC_STATUS_BAD_PARENT;
    if (i > 0 && (tok[i] < 0 || tok[i] >= a.V)) st |= SPEC_STATUS_BAD_TOKEN;
  }
  if (tid == 0) cnt = 0;
  __syncthreads();
  for (int i = tid; i < N; i += kThreads) {
    int d = 0, v = i;
    while (v != 0) {  // parents strictly decrease, so this ends within i steps
      const int pv = par[v];
      if (pv < 0 || pv >= v) {
        d = -1;
        break;
      }
      v = pv;
      ++d;
    }
    dep[i] = static_cast<int16_t>(d);
  }
  __syncthreads();
  for (int i = tid + 1; i < N; i += kThreads) {
    const int p = par[i];
    if (p >= 0 && p < i && dep[p] >= 0) {
      has_child[p] = 1;
      if (dep[p] < a.max_depth && tok[i] >= 0 && tok[i] < a.V) atomicAdd(&testable_child[p], 1);
    }
  }
  __syncthreads();
  for (int i = tid; i < N; i += kThreads) {
    if (testable_child[i] && !bad_t) {
      raw[atomicAdd(&cnt, 1)] = static_cast<int16_t>(i);
    } else {
      TreeRec* rec = a.recs + static_cast<size_t>(b) * N + i;
      uint32_t fl = kRecDetached;
      if (dep[i] >= 0) fl = kRecDefer | (has_child[i] && dep[i] >= a.max_depth ? kRecDepth : 0u);
      if (bad_t) fl = kRecBad;
      rec->accepted = -1;
      rec->flags = fl;
      rec->nmp = 0.f;
      rec->nmq = 0.f;
      rec->fa = 1.f;
      rec->fb = 0.f;
    }
  }
  if (st) atomicOr(a.status, st);
  __syncthreads();
  // order: more children to test first (more possible residual passes), then
  // node index -- one key per listed node, larger first, all keys distinct
  for (int i = tid; i < cnt; i += kThreads) {
    const int ni = raw[i];
    order_key[i] = testable_child[ni] * kMaxTreeNodes + (kMaxTreeNodes - 1 - ni);
  }
  __syncthreads();
  for (int i = tid; i < cnt; i += kThreads) {
    const int mine = order_key[i];
    int r = 0;
#pragma unroll 8
    for (int t = 0; t < cnt; ++t) r += order_key[t] > mine ? 1 : 0;
    list[r] = raw[i];
  }
  if (tid == 0) base = static_cast<int>(atomicAdd(a.work_count, static_cast<uint32_t>(cnt)));
  __syncthreads();
  const int cap = a.B * N;  // the list's length; the count is zero on entry
  for (int i = tid; i < cnt; i += kThreads)
    if (base + i < cap) a.work_list[base + i] = b * N + list[i];
}

// One cluster of kTreeCl CTAs per node with children to test (the list
// tree_plan_kernel built), clusters looping over the list.
template <int DT>
__global__ void __launch_bounds__(kThreads, 3) tree_node_kernel(const TreeSampleArgs a) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ TreeShm sh;
  constexpr int E = Elt<DT>::kBytes;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int ncl = gridDim.x / kTreeCl;
  const int cid = blockIdx.x / kTreeCl;
  const uint32_t sp = smem_addr(dyn);
  const uint32_t sq = sp + static_cast<uint32_t>(a.slice) * E;
  const int lo = rank * a.slice;
  const int len = max(0, min(a.V, lo + a.slice) - lo);
  const int lenv = (len + Elt<DT>::kPerVec - 1) / Elt<DT>::kPerVec * Elt<DT>::kPerVec;  // whole vectors
  const int total = min(static_cast<int>(*a.work_count), a.B * a.N);
  if (threadIdx.x == 0) {
    mbar_init(&sh.bar[0], 1);
    mbar_init(&sh.bar[1], 1);
    fence_mbar_init();
    sh.timed_out = 0;
  }
  __syncthreads();
  uint32_t php = 0, phq = 0;
  int round = 0;
  // the first round takes items cid; later items are claimed from a shared
  // counter, one ahead, during each node's first cluster round
  int kpar = 0;
  for (int idx = cid; idx < total; ++kpar) {
    const int64_t g = a.work_list[idx];
    if (g < 0 || g >= static_cast<int64_t>(a.B) * a.N) break;  // uniform across the cluster
    const int b = static_cast<int>(g / a.N), j = static_cast<int>(g % a.N);
    const int32_t* tok = a.tokens + static_cast<size_t>(b) * a.N;
    const float* uni = a.uniforms + static_cast<size_t>(b) * a.N;
    const float c = tree_c(a, b);
    TreeRec* rec = a.recs + g;
    const unsigned char* pfull = static_cast<const unsigned char*>(a.logits) + static_cast<size_t>(g) * a.V * E;
    const unsigned char* qfull = static_cast<const unsigned char*>(a.draft) + static_cast<size_t>(g) * a.V * E;
    // both rows are needed: start their copies before the tree bookkeeping
    if (a.aligned && threadIdx.x == 0)
      stage_issue(sh, pfull + static_cast<size_t>(lo) * E, qfull + static_cast<size_t>(lo) * E,
                  static_cast<uint32_t>(len) * E, true, sp, sq);
    stage_parents(a, sh, b);
    collect_children(a, sh, tok, j, true);
    const int nk = sh.nk;
    for (int i = threadIdx.x; i < min(nk, kPre); i += kThreads) {
      const int x = tok[sh.kids[i]];
      sh.kl[i] = Elt<DT>::value(Elt<DT>::bits_at(pfull, x));
      sh.kd[i] = Elt<DT>::value(Elt<DT>::bits_at(qfull, x));
      sh.ku[i] = uni[sh.kids[i]];
    }
    stage_rows<DT>(a, sh, pfull + static_cast<size_t>(lo) * E, qfull + static_cast<size_t>(lo) * E, len, true,
                   sp, sq, php, phq, true);
    int slot = round++ & 1;
    if (rank == 0 && threadIdx.x == 0) sh.next[kpar & 1] = ncl + static_cast<int>(atomicAdd(a.work_next, 1u));
    slice_stats<DT>(sh, sp, sq, lenv, a.wchunk, true, c, slot);  // (its cluster barrier publishes sh.next)
    if (threadIdx.x == 0)
      sh.nextl = static_cast<int>(ld_cluster_u32(mapa_shared(smem_addr(&sh.next[kpar & 1]), 0)));
    uint32_t rflags = 0;
    int accepted = -1;
    bool cz = true;
    float fa = 1.f, fb = 0.f, nmp = 0.f, nmq = 0.f;
    const float mp = sh.gm[0], mq = sh.gm[1];
    if (sh.gbad || mp == -INFINITY || mq == -INFINITY) {
      rflags |= kRecBad;
    } else {
      nmp = -mp * c;
      nmq = -mq * c;
      const DF zp = sh.gz[0], zq = sh.gz[1];  // each at least 1: the maximum's own mass
      DF cc{0.f, 0.f}, W{1.f, 0.f};
      for (int i = 0; i < nk; ++i) {
        const int child = sh.kids[i];
        if (threadIdx.x == 0) {
          float lx, dx, uf;
          if (i < kPre) {
            lx = sh.kl[i];
            dx = sh.kd[i];
            uf = sh.ku[i];
          } else {
            const int x = tok[child];
            lx = Elt<DT>::value(Elt<DT>::bits_at(pfull, x));
            dx = Elt<DT>::value(Elt<DT>::bits_at(qfull, x));
            uf = uni[child];
          }
          // u q(x) W < p(x) - cc q(x) with p(x) = ep / zp and q(x) = eq / zq,
          // both sides multiplied by zp zq > 0
          const float ep = ex2_approx(fmaf(lx, c, nmp)), eq = ex2_approx(fmaf(dx, c, nmq));
          const DF lhs = df_mulf(df_mulf(df_mul(W, zp), uf), eq);
          const DF rhs = df_sub(df_mulf(zq, ep), df_mulf(df_mul(cc, zp), eq));
          sh.accept = df_gt(rhs, lhs);
        }
        __syncthreads();
        if (sh.accept) {
          accepted = child;
          break;
        }
        cc = df_add(cc, W);
        fa = __frcp_rn(df_f(zp));
        fb = __fdiv_rn(df_f(cc), df_f(zq));
        slice_pass<DT, 1>(sh, sp, sq, lenv, a.wchunk, true, c, nmp, nmq, fa, fb);
        slot = round++ & 1;
        if (threadIdx.x == 0) {
          DF sum = sh.wsum[0][0];
          sh.wc[0] = sum;
          for (int w = 1; w < kWarps; ++w) {
            sh.wc[w] = sh.wsum[w][0];
            sum = df_add(sum, sh.wsum[w][0]);
          }
          sh.red[slot][0] = sum.hi;
          sh.red[slot][1] = sum.lo;
        }
        cluster_sum(sh, slot);
        const DF wn = sh.gsum;
        if (df_pos(wn)) {
          W = wn;
          cz = false;
        } else {  // residual of mass zero: back to p
          W = DF{1.f, 0.f};
          cc = DF{0.f, 0.f};
          cz = true;
        }
      }
      if (accepted < 0 && threadIdx.x < kWarps) {
        // the c = 0 residual: this CTA's target masses, rescaled to the row maximum
        const float m0 = sh.mloc[0];
        const float scale = m0 == -INFINITY ? 0.f : ex2_approx((m0 - mp) * c);
        const DF w = cz ? df_mulf(sh.zc[threadIdx.x], scale) : sh.wc[threadIdx.x];
        rec->chunk[rank * kWarps + threadIdx.x][0] = w.hi;
        rec->chunk[rank * kWarps + threadIdx.x][1] = w.lo;
      }
    }
    if (rank == 0 && threadIdx.x == 0) {
      rec->accepted = accepted;
      rec->flags = rflags;
      rec->nmp = nmp;
      rec->nmq = nmq;
      rec->fa = cz ? 1.f : fa;
      rec->fb = cz ? 0.f : fb;
    }
    __syncthreads();  // every read of this node's slices and of sh.par is done
    idx = sh.nextl;
  }
  if (sh.timed_out && threadIdx.x == 0) {  // let copies still in flight land before the CTA leaves
    mbar_wait_bounded(&sh.bar[0], php ^ 1u);
    mbar_wait_bounded(&sh.bar[1], phq ^ 1u);
  }
  cluster.sync();  // no CTA leaves while a peer may still read its shared memory
}

// One cluster per tree: follow the accepted children from the root (every
// CTA walks the same records), sum the stop node's p if its node pass left
// that to the walk, then rank 0 draws the correction.
template <int DT>
__global__ void __launch_bounds__(kThreads, 1) tree_walk_kernel(const TreeSampleArgs a) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ TreeShm sh;
  constexpr int E = Elt<DT>::kBytes;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / kTreeCl;
  const int tid = threadIdx.x;
  const int D = a.max_depth + 1;
  int32_t* otok = a.out_tokens + static_cast<size_t>(b) * D;
  int32_t* opath = a.out_path + static_cast<size_t>(b) * D;
  const int32_t* tok = a.tokens + static_cast<size_t>(b) * a.N;
  // every node's outcome in one round of loads; thread 0 then walks them here
  __shared__ int16_t w_acc[kMaxTreeNodes];
  __shared__ uint8_t w_fl[kMaxTreeNodes];
  __shared__ int16_t w_path[kMaxTreeNodes];
  const TreeRec* trec = a.recs + static_cast<size_t>(b) * a.N;
  for (int i = tid; i < a.N; i += kThreads) {
    const int acc = trec[i].accepted;
    w_acc[i] = static_cast<int16_t>(acc > i && acc < a.N ? acc : -1);  // a child's id exceeds its parent's
    w_fl[i] = static_cast<uint8_t>(trec[i].flags | (acc >= 0 && !(acc > i && acc < a.N) ? kRecBad : 0u));
  }
  if (tid == 0) {
    mbar_init(&sh.bar[0], 1);
    mbar_init(&sh.bar[1], 1);
    fence_mbar_init();
    sh.timed_out = 0;
    sh.has_child = 0;
  }
  __syncthreads();
  if (tid == 0) {
    int v = 0, n = 0, ok = 1;
    uint32_t st = 0;
    for (int it = 0; it <= a.max_depth; ++it) {
      const uint32_t fl = w_fl[v];
      const int acc = w_acc[v];
      if (fl & (kRecBad | kRecDetached)) {
        ok = 0;
        st |= SPEC_STATUS_BAD_ROW;
        break;
      }
      if (acc >= 0) {
        if (n >= a.max_depth) {  // not reachable: children at max_depth are never tested
          ok = 0;
          break;
        }
        w_path[n++] = static_cast<int16_t>(acc);
        v = acc;
        continue;
      }
      if (fl & kRecDepth) st |= SPEC_STATUS_DEPTH;
      sh.has_child = (fl & kRecDefer) != 0;
      break;
    }
    if (rank == 0 && st) atomicOr(a.status, st);
    sh.walk_v = v;
    sh.walk_n = n;
    sh.walk_ok = ok;
  }
  __syncthreads();
  const int v = sh.walk_v, n = sh.walk_n;
  bool ok = sh.walk_ok != 0;
  if (rank == 0)
    for (int i = tid; i < D; i += kThreads) {
      if (i < n) {
        opath[i] = w_path[i];
        otok[i] = tok[w_path[i]];
      } else {
        opath[i] = -1;
        if (i > n) otok[i] = -1;
      }
    }
  const bool local = ok && sh.has_child;
  float nmp_l = 0.f;
  if (local) {  // stop distribution p of a node whose pass only marked it
    const size_t g = static_cast<size_t>(b) * a.N + v;
    const uint32_t sp = smem_addr(dyn);
    const int lo = rank * a.slice;
    const int len = max(0, min(a.V, lo + a.slice) - lo);
    uint32_t php = 0, phq = 0;
    stage_rows<DT>(a, sh, static_cast<const unsigned char*>(a.logits) + (g * a.V + lo) * E, nullptr, len, false,
                   sp, sp, php, phq, false);
    slice_stats<DT>(sh, sp, sp, (len + Elt<DT>::kPerVec - 1) / Elt<DT>::kPerVec * Elt<DT>::kPerVec, a.wchunk, false,
                    tree_c(a, b), 0);
    const float mp = sh.gm[0];
    if (sh.gbad || mp == -INFINITY) {
      ok = false;
      if (rank == 0 && tid == 0) atomicOr(a.status, SPEC_STATUS_BAD_ROW);
    } else {
      if (tid < kWarps) {  // this CTA's chunk sums, rescaled to the row maximum, for rank 0's draw
        const float m0 = sh.mloc[0];
        const float scale = m0 == -INFINITY ? 0.f : ex2_approx((m0 - mp) * tree_c(a, b));
        sh.wc[tid] = df_mulf(sh.zc[tid], scale);
      }
      nmp_l = -mp * tree_c(a, b);
    }
    if (sh.timed_out && tid == 0) mbar_wait_bounded(&sh.bar[0], php ^ 1u);
    cluster.sync();  // every CTA's chunk sums are in its shared memory
  }
  if (rank == 0) {
    if (ok) {
      draw_at<DT>(a, sh, b, v, n, local, nmp_l, 0.f, 1.f, 0.f);
    } else if (tid == 0) {
      otok[n] = -1;
      a.out_n[b] = n;
    }
  }
  if (blockIdx.x == 0 && tid == 0) {  // the node pass has read both: zero for the next call
    *a.work_count = 0u;
    *a.work_next = 0u;
  }
  cluster.sync();  // no CTA leaves while a peer may still read its shared memory
}

cudaLaunchConfig_t cluster_config(cudaLaunchAttribute* attr, size_t smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kTreeCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Shared-memory opt-in and cluster occupancy of the node kernel, per device
// and dtype: the last shared-memory size set and the clusters that fit.
constexpr int kTreeMaxDevices = 64;
struct TreeLaunchCache {
  int smem = -1;
  int clusters = 0;
};
std::mutex g_tree_mu;
TreeLaunchCache g_tree_cache[kTreeMaxDevices][2];

template <int DT>
int launch_tree_t(const TreeSampleArgs& a, cudaStream_t st) {
  const size_t smem = tree_smem_bytes(DT, a.slice);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kTreeMaxDevices) return cudaErrorInvalidDevice;
  auto node_k = tree_node_kernel<DT>;
  auto walk_k = tree_walk_kernel<DT>;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(attr, smem, st);
  int max_clusters = 0;
  {
    std::lock_guard<std::mutex> lock(g_tree_mu);
    TreeLaunchCache& c = g_tree_cache[dev][DT];
    if (c.smem != static_cast<int>(smem)) {
      e = cudaFuncSetAttribute(node_k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(walk_k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      cfg.gridDim = dim3(kTreeCl);
      int ncl = 0;
      e = cudaOccupancyMaxActiveClusters(&ncl, node_k, &cfg);
      if (e != cudaSuccess) return e;
      if (ncl < 1) return cudaErrorInvalidConfiguration;
      c.smem = static_cast<int>(smem);
      c.clusters = ncl;
    }
    max_clusters = c.clusters;
  }
  tree_plan_kernel<<<a.B, kThreads, 0, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t nodes = static_cast<int64_t>(a.B) * a.N;
  const int clusters = static_cast<int>(nodes < max_clusters ? nodes : max_clusters);
  cfg.gridDim = dim3(clusters * kTreeCl);
  e = cudaLaunchKernelEx(&cfg, node_k, a);
  if (e == cudaSuccess) {
    cfg.gridDim = dim3(static_cast<unsigned>(a.B) * kTreeCl);
    e = cudaLaunchKernelEx(&cfg, walk_k, a);
  }
  if (e != cudaSuccess) cudaMemsetAsync(a.work_count, 0, 2 * sizeof(uint32_t), st);  // the walk did not reset them
  return e;
}

}  // namespace

size_t tree_smem_bytes(int dtype, int slice) {
  return 2 * static_cast<size_t>(slice) * (dtype == DT_BF16 ? 2 : 4);
}

int launch_tree_sample(const TreeSampleArgs& a, int dtype, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return dtype == DT_BF16 ? launch_tree_t<DT_BF16>(a, st) : launch_tree_t<DT_F32>(a, st);
}

}  // namespace specv
