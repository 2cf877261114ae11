// kv_kernel.cu -- the KV-cache keep list after a verification pass.
//
// "Towards Green Text Generation: Memory-Based Speculative Decoding",
// section 2.4 (KV-cached regime): on rejection the cache is cut back to the
// accepted prefix.  Edge Inference Notes, "One decode round, end to end": the
// longest agreed path of the token tree is committed and the other branches
// collapse.  For every sequence this kernel lists, per kept entry, the slot
// it occupies after the pass (the root's and the path nodes' entries, in
// path order) and the slot it takes once the cache is cut back (consecutive
// positions from the root's), translated through a block table when the
// cache is paged.
//
// One warp per sequence: a first sweep over the kept entries checks the path
// and every block lookup (a bad sequence is left out whole), a second writes
// the list and its -1 padding.  The work is a few hundred bytes per
// sequence; the launch is latency-bound by design.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace specv {
namespace {

constexpr int kKvWarps = 8;
constexpr unsigned kFull = 0xffffffffu;

// Node id of the d-th kept entry: the root for d = 0, then the path's nodes
// (a chain's node d is its d-th position).
__device__ __forceinline__ long long kept_node(const KvArgs& a, int b, int d) {
  if (d == 0) return 0;
  if (a.path == nullptr) return d;
  return a.path[(size_t)b * a.path_stride + (d - 1)];
}

// Physical slot of logical position pos of sequence b; -1 if the lookup is
// out of range.
__device__ __forceinline__ long long slot_of(const KvArgs& a, int b, long long pos) {
  if (a.block_table == nullptr) return pos;
  const long long blk = pos / a.block_size;
  if (blk >= a.max_blocks) return -1;
  const int phys = a.block_table[(size_t)b * a.max_blocks + blk];
  if (phys < 0) return -1;
  const long long s = (long long)phys * a.block_size + pos % a.block_size;
  return s > INT32_MAX ? -1 : s;
}

__global__ void __launch_bounds__(kKvWarps * 32) kv_compact_kernel(KvArgs a) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kKvWarps + (threadIdx.x >> 5);
  if (b >= a.B) return;  // whole warps leave together
  const int n = a.n[b];
  const long long base = a.base[b];
  bool ok = n >= 0 && (long long)n + 1 <= a.max_keep && base >= 0 && base + n + 1 <= INT32_MAX &&
            (a.path == nullptr || n <= a.path_stride);
  int moves = 0;
  long long carry = 0;  // node of the entry before this sweep's first
  for (int d0 = 0; ok && d0 <= n; d0 += 32) {
    const int d = d0 + lane;
    const bool live = d <= n;
    const long long node = live ? kept_node(a, b, d) : 0;
    long long prev = __shfl_up_sync(kFull, node, 1);
    if (lane == 0) prev = carry;
    bool good = true;
    if (live) {
      // strictly above the entry before (the root is 0), hence >= d
      if (d > 0 && node <= prev) good = false;
      const long long src = base + node, dst = base + d;
      if (good && (src > INT32_MAX || slot_of(a, b, src) < 0 || slot_of(a, b, dst) < 0)) good = false;
    }
    const unsigned mv = __ballot_sync(kFull, live && good && node != d);
    if (lane == 0) moves += __popc(mv);
    ok = __all_sync(kFull, good);
    carry = __shfl_sync(kFull, node, 31);
  }
  moves = __shfl_sync(kFull, moves, 0);
  int32_t* src_row = a.out_src + (size_t)b * a.max_keep;
  int32_t* dst_row = a.out_dst + (size_t)b * a.max_keep;
  for (int d = lane; d < a.max_keep; d += 32) {
    int32_t s = -1, t = -1;
    if (ok && d <= n) {
      s = (int32_t)slot_of(a, b, base + kept_node(a, b, d));
      t = (int32_t)slot_of(a, b, base + d);
    }
    src_row[d] = s;
    dst_row[d] = t;
  }
  if (lane == 0) {
    a.out_new_len[b] = ok ? (int32_t)(base + n + 1) : -1;
    if (a.out_moves) a.out_moves[b] = ok ? moves : 0;
    if (!ok && a.status) atomicOr(a.status, SPEC_STATUS_BAD_KV);
  }
}

}  // namespace

int launch_kv_compact(const KvArgs& a, void* stream) {
  const int grid = (a.B + kKvWarps - 1) / kKvWarps;
  kv_compact_kernel<<<grid, kKvWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return (int)cudaGetLastError();
}

}  // namespace specv
