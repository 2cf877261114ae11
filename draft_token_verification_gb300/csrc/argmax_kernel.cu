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
// Both reduce to one argmax per row (lowest index on ties) followed by a tiny
// per-sequence walk.  Each row is split over several CTAs that stream their
// slice once with 16-byte non-allocating loads; a CTA's (value, index) winner
// is folded into the row's slot with one 64-bit atomicMax on an order-
// preserving packing; the last CTA of a sequence (atomic ticket, no
// spin-wait) does the walk, writes the outputs and re-zeroes the slots.
#include <cuda_runtime.h>
#include <math.h>

#include "device_common.cuh"

namespace specv {

namespace {

constexpr int kUnroll = 8;  // 16-byte loads in flight per thread

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
  int depth[kMaxTreeNodes];
  unsigned char agreed[kMaxTreeNodes];
};

}  // namespace

template <int DT, bool TREE>
__global__ void __launch_bounds__(kThreads) argmax_kernel(const ArgmaxArgs a) {
  using E = Elt<DT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = static_cast<int>(blockIdx.x) / a.splits;
  const int split = static_cast<int>(blockIdx.x) % a.splits;
  const int b = row / a.R;
  const int lo = min(a.V, split * a.split_len);
  const int hi = min(a.V, lo + a.split_len);
  const unsigned char* base =
      static_cast<const unsigned char*>(a.logits) + static_cast<size_t>(row) * a.V * E::kBytes;

  __shared__ unsigned long long s_best[kWarps];
  __shared__ uint32_t s_nan[kWarps];
  __shared__ int s_last;

  // ---- this thread's best over its vectors: (value, first vector holding it)
  float best = 0.f;
  int best_pos = -1;  // element index of the first vector (or element) holding `best`
  uint32_t nan_seen = 0;
  if (a.aligned) {
    const int nvec = (hi - lo) / E::kPerVec;  // lo, hi are multiples of kPerVec (hi may be V)
    const uint4* vp = reinterpret_cast<const uint4*>(base + static_cast<size_t>(lo) * E::kBytes);
    for (int v0 = tid; v0 < nvec; v0 += kThreads * kUnroll) {
      uint4 x[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + u * kThreads;
        x[u] = v < nvec ? ldg_stream(vp + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + u * kThreads;
        if (v < nvec) {
          float vm = E::value(E::bits_of(x[u], 0));
#pragma unroll
          for (int j = 1; j < E::kPerVec; ++j) vm = max_nan(vm, E::value(E::bits_of(x[u], j)));
          if (vm != vm) {
            nan_seen = 1u;
          } else if (best_pos < 0 || vm > best) {
            best = vm;
            best_pos = lo + v * E::kPerVec;
          }
        }
      }
    }
    // the first element of the winning vector that equals the vector maximum
    if (best_pos >= 0) {
      const uint4 x = ldg_stream(reinterpret_cast<const uint4*>(base + static_cast<size_t>(best_pos) * E::kBytes));
      int j0 = E::kPerVec - 1;
#pragma unroll
      for (int j = E::kPerVec - 1; j >= 0; --j)
        if (E::value(E::bits_of(x, j)) == best) j0 = j;
      best_pos += j0;
    }
  } else {
    for (int t = lo + tid; t < hi; t += kThreads) {
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
    const uint32_t bits = (E::kBytes == 2) ? (__float_as_uint(best) >> 16) : __float_as_uint(best);
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
    const uint32_t total = static_cast<uint32_t>(a.R * a.splits);
    s_last = (atomicAdd(a.tickets + b, 1u) == total - 1u) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ------------------------------------------- last CTA of sequence b: walk
  unsigned long long* slots = a.slots + static_cast<size_t>(b) * a.R;
  if constexpr (!TREE) {
    if (tid == 0) {
      const int k = a.R - 1;
      const int32_t* x = a.tokens + static_cast<size_t>(b) * k;
      int32_t* out = a.out_tokens + static_cast<size_t>(b) * (k + 1);
      int n = k;
      for (int i = 0; i <= k; ++i) {
        const int am = unpack_index(__ldcg(slots + i));
        if (i == k || x[i] != am) {
          out[i] = am;
          n = i;
          break;
        }
        out[i] = am;
      }
      for (int i = n + 1; i <= k; ++i) out[i] = -1;
      a.out_n[b] = n;
    }
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
    if (tid == 0) {
      uint32_t st = 0;
      if (ts.par[0] != -1) st |= SPEC_STATUS_BAD_PARENT;
      ts.agreed[0] = 1;
      ts.depth[0] = 0;
      int best = 0;
      for (int j = 1; j < N; ++j) {
        const int p = ts.par[j];
        ts.agreed[j] = 0;
        ts.depth[j] = 0;
        if (p < 0 || p >= j) {
          st |= SPEC_STATUS_BAD_PARENT;
          continue;
        }
        ts.depth[j] = ts.depth[p] + 1;
        bool ag = ts.agreed[p] && ts.tok[j] == ts.am[p];
        if (ag && ts.depth[j] > a.max_depth) {
          st |= SPEC_STATUS_DEPTH;
          ag = false;
        }
        ts.agreed[j] = ag ? 1 : 0;
        if (ag && ts.depth[j] > ts.depth[best]) best = j;
      }
      const int D = a.max_depth + 1;
      int32_t* ot = a.out_tokens + static_cast<size_t>(b) * D;
      int32_t* op = a.out_path + static_cast<size_t>(b) * D;
      const int len = ts.depth[best];
      for (int i = len + 1; i < D; ++i) { ot[i] = -1; op[i] = -1; }
      ot[len] = ts.am[best];
      if (len < D) op[len] = -1;
      for (int c = best, i = len - 1; c != 0; c = ts.par[c], --i) {
        op[i] = c;
        ot[i] = ts.tok[c];
      }
      a.out_n[b] = len;
      set_status(a.status, st);
    }
  }
  __syncthreads();
  for (int j = tid; j < a.R; j += kThreads) slots[j] = 0ull;
  if (tid == 0) a.tickets[b] = 0u;
}

int launch_argmax(const ArgmaxArgs& a, int dtype, bool tree, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 grid(static_cast<unsigned>(a.B * a.R * a.splits));
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
