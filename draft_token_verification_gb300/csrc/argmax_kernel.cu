// argmax_kernel.cu -- greedy chain and greedy token-tree verification on sm_103a.
//
// Greedy chain ("Towards Green Text Generation: Memory-Based Speculative
// Decoding", section 2.4 "Verifier and Acceptance"): the k+1 target rows are
// compared greedily with the k drafts; the longest prefix equal to the
// target's argmax is accepted, plus the target's own token after it.
// Greedy tree (Edge Inference Notes, post on speculative decoding and
// EAGLE-3, "One decode round, end to end"): the longest root-to-node path
// whose tokens all equal the argmax of their parent's row is committed, plus
// the argmax of its last node's row.
//
// Both reduce to one argmax per row (lowest index on ties, -0 equal to +0)
// followed by a tiny per-sequence walk.  The batch's rows are laid end to end
// as 16-byte vectors and cut into one equal range per CTA, one wave of CTAs
// sized to the GPU; a CTA streams its range once with 16-byte non-allocating
// loads, eight in flight per thread, and folds its (value, index) winner for
// each row piece into the row's slot with one 64-bit atomicMax on an order-
// preserving packing.  A per-sequence ticket counts the vectors folded in; the
// CTA that completes a sequence (no spin-wait) does the walk, writes the
// outputs and re-zeroes the slots.
#include <cuda_runtime.h>

#include <algorithm>
#include <math.h>

#include "device_common.cuh"

namespace specv {

namespace {

constexpr int kUnroll = 8;  // 16-byte loads in flight per thread

// NaN-propagating maximum of two bf16 pairs.
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// (value key, ~index): a larger packing is a larger value, then a lower index.
__device__ __forceinline__ unsigned long long pack_best(uint32_t key, int idx) {
  return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(idx));
}

__device__ __forceinline__ int unpack_index(unsigned long long p) {
  return static_cast<int>(~static_cast<uint32_t>(p & 0xFFFFFFFFull));
}

struct TreeShm {
  int am[kMaxTreeNodes];
  int par[kMaxTreeNodes];
  int tok[kMaxTreeNodes];
};

__device__ __forceinline__ int warp_max_i32(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

}  // namespace

// The walk of sequence b by the CTA that completed it (whole CTA; every
// node or position in parallel, no serial chain of loads).
template <bool TREE>
__device__ __forceinline__ void sequence_walk(const ArgmaxArgs& a, int b) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long* slots = a.slots + static_cast<size_t>(b) * a.R;
  __shared__ int s_red[kWarps];
  if constexpr (!TREE) {
    if (a.first_check) {  // the rejection fast path: one row, the first draft
      if (tid == 0) {
        const int am = unpack_index(__ldcg(slots));
        a.out_tokens[b] = am;
        a.out_n[b] = a.tokens[b] == am ? 1 : 0;
        slots[0] = 0ull;
        a.tickets[b] = 0u;
      }
      return;
    }
    // n = the first position whose draft differs from the target's argmax
    const int k = a.R - 1;
    const int32_t* x = a.tokens + static_cast<size_t>(b) * k;
    int32_t* out = a.out_tokens + static_cast<size_t>(b) * (k + 1);
    int first = k;
    for (int i = tid; i < k; i += kThreads)
      if (x[i] != unpack_index(__ldcg(slots + i))) first = min(first, i);
    first = -warp_max_i32(-first);
    if (lane == 0) s_red[warp] = first;
    __syncthreads();
    int n = k;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) n = min(n, s_red[w]);
    for (int i = tid; i <= k; i += kThreads) out[i] = i <= n ? unpack_index(__ldcg(slots + i)) : -1;
    if (tid == 0) a.out_n[b] = n;
  } else {
    __shared__ TreeShm ts;
    const int N = a.R;
    const int32_t* par = a.parents + static_cast<size_t>(b) * N;
    const int32_t* tok = a.tokens + static_cast<size_t>(b) * N;
    for (int j = tid; j < N; j += kThreads) {
      ts.am[j] = unpack_index(__ldcg(slots + j));
      ts.par[j] = par[j];
      ts.tok[j] = tok[j];
    }
    __syncthreads();
    // node j is agreed iff every node on its path from the root has a valid
    // parent (p < j) and a token equal to its parent's argmax, and it lies at
    // depth <= max_depth; an agreed-path node at max_depth + 1 is reported.
    // Best: the deepest agreed node, the lowest index among equals.
    uint32_t st = 0;
    int key = -1;
    for (int j = tid; j < N; j += kThreads) {
      if (j == 0) {
        if (ts.par[0] != -1) st |= SPEC_STATUS_BAD_PARENT;
        key = max(key, (0 << 16) | 0xFFFF);
        continue;
      }
      const int pj = ts.par[j];
      if (pj < 0 || pj >= j) st |= SPEC_STATUS_BAD_PARENT;
      bool ok = true;  // every node from j up has a valid parent and matches its argmax
      int d = 0;       // edges walked from j
      for (int c = j; c != 0;) {
        const int p = ts.par[c];
        // an invalid parent, or j deeper than max_depth + 1 (neither kept nor reported)
        if (p < 0 || p >= c || d > a.max_depth) {
          ok = false;
          break;
        }
        ok = ok && ts.tok[c] == ts.am[p];
        ++d;
        c = p;
      }
      if (ok && d > a.max_depth) {
        if (d == a.max_depth + 1) st |= SPEC_STATUS_DEPTH;
        ok = false;
      }
      if (ok) key = max(key, (d << 16) | (0xFFFF - j));
    }
    if (st) set_status(a.status, st);
    key = warp_max_i32(key);
    if (lane == 0) s_red[warp] = key;
    __syncthreads();
    if (tid == 0) {
      int bk = -1;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) bk = max(bk, s_red[w]);
      const int best = 0xFFFF - (bk & 0xFFFF);
      const int D = a.max_depth + 1;
      int32_t* ot = a.out_tokens + static_cast<size_t>(b) * D;
      int32_t* op = a.out_path + static_cast<size_t>(b) * D;
      const int len = bk >> 16;
      for (int i = len + 1; i < D; ++i) { ot[i] = -1; op[i] = -1; }
      ot[len] = ts.am[best];
      if (len < D) op[len] = -1;
      for (int c = best, i = len - 1; c != 0; c = ts.par[c], --i) {
        op[i] = c;
        ot[i] = ts.tok[c];
      }
      a.out_n[b] = len;
    }
  }
  __syncthreads();
  for (int j = tid; j < a.R; j += kThreads) slots[j] = 0ull;
  if (tid == 0) a.tickets[b] = 0u;
}

template <int DT, bool TREE>
__global__ void __launch_bounds__(kThreads) argmax_kernel(const ArgmaxArgs a) {
  using E = Elt<DT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V, nvr = a.nvr;
  // this CTA's range of row vectors (rows laid end to end)
  const long long units = static_cast<long long>(a.B) * a.R * nvr;
  const long long u0 = static_cast<long long>(blockIdx.x) * units / gridDim.x;
  const long long u1 = (static_cast<long long>(blockIdx.x) + 1) * units / gridDim.x;
  const uint32_t seq_units = static_cast<uint32_t>(a.R) * static_cast<uint32_t>(nvr);

  __shared__ unsigned long long s_best[kWarps];
  __shared__ uint32_t s_nan[kWarps];
  __shared__ int s_last;

  for (long long us = u0; us < u1;) {
    // the piece of one row: row vectors [v_lo, v_hi)
    const int row = static_cast<int>(us / nvr);
    const long long rbeg = static_cast<long long>(row) * nvr;
    const long long ue = min(u1, rbeg + nvr);
    const int v_lo = static_cast<int>(us - rbeg), v_hi = static_cast<int>(ue - rbeg);
    us = ue;
    const int b = row / a.R;
    const unsigned char* base =
        static_cast<const unsigned char*>(a.logits) + static_cast<size_t>(row) * V * E::kBytes;

    // ---- this thread's best: (value, its first index), vectors in index order
    float best = 0.f;
    int best_pos = -1;
    uint32_t nan_seen = 0;
    if (a.aligned) {  // whole 16-byte vectors (V is a multiple of kPerVec)
      const uint4* vp = reinterpret_cast<const uint4*>(base);
      // Branch-free fold: the first vector whose maximum is the largest so
      // far (strictly, so an earlier vector keeps a tie) is kept with its
      // bits; the element's place in it is found once at the end.  A vector
      // holding NaN is never kept and leaves nan_acc NaN.
      float bv = -INFINITY, nan_acc = 0.f;
      int bidx = -1;
      uint4 bx = make_uint4(0u, 0u, 0u, 0u);
      auto fold = [&](const uint4& x, int v) {
        float vm;
        if constexpr (DT == DT_BF16) {  // packed: three bf16x2 maxima, then the two halves
          const uint32_t m2 = bmax2_nan(bmax2_nan(x.x, x.y), bmax2_nan(x.z, x.w));
          vm = max_nan(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
        } else {
          vm = E::value(E::bits_of(x, 0));
#pragma unroll
          for (int j = 1; j < E::kPerVec; ++j) vm = max_nan(vm, E::value(E::bits_of(x, j)));
        }
        nan_acc = max_nan(nan_acc, vm);
        const bool take = vm > bv || (bidx < 0 && vm == vm);
        bv = take ? vm : bv;
        bidx = take ? v : bidx;
        bx.x = take ? x.x : bx.x;
        bx.y = take ? x.y : bx.y;
        bx.z = take ? x.z : bx.z;
        bx.w = take ? x.w : bx.w;
      };
      int v0 = v_lo + tid;
      for (; v0 + (kUnroll - 1) * kThreads < v_hi; v0 += kThreads * kUnroll) {  // every load in range
        uint4 x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) x[u] = ldg_stream(vp + v0 + u * kThreads);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) fold(x[u], v0 + u * kThreads);
      }
      if (v0 < v_hi) {  // the last batch, in part
        uint4 x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + u * kThreads;
          x[u] = v < v_hi ? ldg_stream(vp + v) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (v0 + u * kThreads < v_hi) fold(x[u], v0 + u * kThreads);
      }
      nan_seen = nan_acc != nan_acc ? 1u : 0u;
      if (bidx >= 0) {
        int j0 = E::kPerVec - 1;
#pragma unroll
        for (int j = E::kPerVec - 1; j >= 0; --j)
          if (E::value(E::bits_of(bx, j)) == bv) j0 = j;
        best = bv;
        best_pos = bidx * E::kPerVec + j0;
      }
    } else {
      const int hi = min(V, v_hi * E::kPerVec);
      for (int t = v_lo * E::kPerVec + tid; t < hi; t += kThreads) {
        const float v = E::value(E::bits_at(base, t));
        if (v != v) {
          nan_seen = 1u;
        } else if (best_pos < 0 || v > best) {
          best = v;
          best_pos = t;
        }
      }
    }
    unsigned long long mine = 0ull;
    if (best_pos >= 0) {
      // -0 and +0 compare equal: both take the key of +0
      const uint32_t bits = best == 0.f ? 0u
                            : (E::kBytes == 2) ? (__float_as_uint(best) >> 16) : __float_as_uint(best);
      mine = pack_best(E::key(bits), best_pos);
    }
    mine = warp_max_u64(mine);
    nan_seen = warp_max_u32(nan_seen);
    if (lane == 0) { s_best[warp] = mine; s_nan[warp] = nan_seen; }
    __syncthreads();
    if (tid == 0) {
      unsigned long long m = 0ull;
      uint32_t nn = 0;
      for (int w = 0; w < kWarps; ++w) { m = s_best[w] > m ? s_best[w] : m; nn |= s_nan[w]; }
      if (nn) set_status(a.status, SPEC_STATUS_BAD_ROW);
      if (m) atomicMax(a.slots + row, m);
      __threadfence();
      const uint32_t mine_units = static_cast<uint32_t>(v_hi - v_lo);
      s_last = (atomicAdd(a.tickets + b, mine_units) + mine_units == seq_units) ? 1 : 0;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      sequence_walk<TREE>(a, b);
    }
  }
}

// Streaming multiprocessors of the current device (cached per device).
int num_sms() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 148;
  if (dev < 64) cache[dev] = sms;
  return sms;
}

int launch_argmax(const ArgmaxArgs& args, int dtype, bool tree, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* kern = dtype == DT_BF16 ? (tree ? reinterpret_cast<const void*>(argmax_kernel<DT_BF16, true>)
                                              : reinterpret_cast<const void*>(argmax_kernel<DT_BF16, false>))
                                      : (tree ? reinterpret_cast<const void*>(argmax_kernel<DT_F32, true>)
                                              : reinterpret_cast<const void*>(argmax_kernel<DT_F32, false>));
  // one wave: resident CTAs per SM x SMs, at most one CTA per 256 row vectors
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const long long units = static_cast<long long>(args.B) * args.R * args.nvr;
  long long g = static_cast<long long>(num_sms()) * per_sm;
  g = std::min(g, (units + 255) / 256);
  ArgmaxArgs a = args;
  a.grid = static_cast<int>(std::max(1LL, g));
  const dim3 grid(static_cast<unsigned>(a.grid));
  if (dtype == DT_BF16) {
    if (tree) argmax_kernel<DT_BF16, true><<<grid, kThreads, 0, st>>>(a);
    else argmax_kernel<DT_BF16, false><<<grid, kThreads, 0, st>>>(a);
  } else {
    if (tree) argmax_kernel<DT_F32, true><<<grid, kThreads, 0, st>>>(a);
    else argmax_kernel<DT_F32, false><<<grid, kThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace specv
