// internal.h -- declarations shared by the C ABI (api.cu) and the kernels:
// dtype codes, the workspace layout and the kernel argument blocks.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "spec_verify.h"

namespace specv {

constexpr int DT_F32 = 0;
constexpr int DT_BF16 = 1;

constexpr int kThreads = 256;           // threads per CTA in every kernel
constexpr int kWarps = kThreads / 32;
constexpr int kWindow = 512;            // exact-value histogram bins per row
constexpr int kMaxK = 31;
constexpr int kMaxTreeNodes = 1024;

constexpr int MODE_SAMPLE = 0;          // speculative-sampling verification
constexpr int MODE_PROBS = 1;           // write filtered probabilities

// The kept set and normaliser of one filtered row: token j of key (value
// order) `key` is kept iff all_kept, or key > kstar, or key == kstar and
// j < tie_cut; its probability is 2^(l c - K) * inv_z.
struct RowState {
  float c;               // log2(e) / T
  float K;               // lattice exponent (an integer) of the row
  float m;               // row maximum
  uint32_t kmax;         // key of m
  uint32_t kstar;
  int32_t tie_cut;
  float inv_z;           // 1 / mass of the kept set
  float zkept;
  int32_t all_kept;
  int32_t covered;       // the kept set was decided from candidate vectors
  int32_t bad;
};

// Sampling runs as three launches.  The stream kernel reads every row once
// and leaves a RowHdr and its candidate tags; the tail kernel decides each
// row's kept set from them (RowPub) and, in the last CTA of a sequence, the
// accepted prefix n; the draw kernel draws the token at position n.
constexpr int kTagsPerWarp = 1024;      // candidate tags per warp segment handed to the tail kernel
constexpr int kRowTags = kWarps * kTagsPerWarp;

// One row after the stream kernel.
struct RowHdr {
  float m;               // row maximum
  float K;               // lattice exponent
  float zhi, zlo;        // sum of 2^(l c - K) over the row, as a double-float
  uint32_t kmax;         // key of m
  uint32_t klo;          // every tag list is complete at and above this key
  uint32_t xbits;        // the row's value at the draft token (draft positions)
  int32_t bad;           // bad temperature, no finite maximum, or |m c| >= 2^30
  uint32_t ntags[kWarps];  // tags at or above klo handed over per warp segment
};

// One row after the tail kernel: its kept set, its probability at the draft
// token and, for target rows, the row vectors holding its kept tokens in
// index order (nlist = kPubReread when they are not listed).
constexpr int kPubList = 1024;
constexpr uint32_t kPubReread = 0xFFFFFFFFu;
struct RowPub {
  RowState rs;
  float xprob;
  uint32_t nlist;
  uint32_t pad[2];
  uint32_t list[kPubList];
};

// Chunks of the draw at the first rejection: one CTA each.  A chunk's record:
// its residual and p sums (two double-floats), then its per-warp sums
// (kWarps residual, kWarps p).
constexpr int kMaxDrawChunks = 16;
constexpr int kChunkRec = 4 + 2 * kWarps;  // floats

// Token-tree sampling verification runs one thread-block cluster of kTreeCl
// CTAs per node: CTA r of the cluster holds elements [r*slice, (r+1)*slice)
// of the node's target and draft rows in shared memory, and warp w of it the
// chunk [w*wchunk, (w+1)*wchunk) of that slice.  A node leaves one TreeRec:
// the first accepted child, or the residual it stops with and that
// residual's per-chunk sums (the draw's first level); a node without children
// to test leaves only its flags.
constexpr int kTreeCl = 8;
constexpr int kTreeChunks = kTreeCl * kWarps;
constexpr size_t kTreeSmemMax = 200 * 1024;  // dynamic shared memory of one tree CTA
constexpr uint32_t kRecBad = 1u;        // a non-finite row at this node
constexpr uint32_t kRecDepth = 2u;      // children not tested: the node is at max_depth
constexpr uint32_t kRecDetached = 4u;   // a malformed parent on the way to the root
constexpr uint32_t kRecDefer = 8u;      // no child to test: the stop residual is p, summed by the walk
struct TreeRec {
  int32_t accepted;      // node id of the accepted child, or -1
  uint32_t flags;        // kRec*
  float nmp, nmq;        // -max * log2(e) / T of the target and draft rows
  float fa, fb;          // stop residual weight: max(0, 2^(l c + nmp) fa - 2^(d c + nmq) fb)
  int32_t pad[2];
  float chunk[kTreeChunks][2];  // sums of that weight per (CTA, warp) chunk, double-float (hi, lo)
};
// The tree draw scans the chunk sums with one warp, two chunks per lane.
static_assert(kTreeChunks == 2 * 32, "the tree draw reads exactly two chunk sums per lane of one warp");

// Workspace layout (byte offsets), identical for every call with the same
// (B, k).  Tickets are zero between calls; everything else is written before
// it is read within a call (the status word collects sticky bits until
// spec_get_status clears it).
struct WsLayout {
  size_t status;      // uint32 status word (sticky bits)
  size_t s_tickets;   // uint32[B]  rows finished per sequence, tail kernel
  size_t d_tickets;   // uint32[B]  chunks finished per sequence, draw kernel
  size_t work;        // uint32[2]  fused stream/tail kernel: next work item, CTAs finished
  size_t done;        // uint32[rows]  fused kernel: a row's stream part is published
  size_t hdrs;        // RowHdr[rows]
  size_t tags;        // uint32[rows][kRowTags]
  size_t pubs;        // RowPub[rows]
  size_t csums;       // float[B][kMaxDrawChunks][kChunkRec]  per-chunk draw sums
  size_t g_slots;     // uint64[B*(k+1)]  packed (value key, ~index) per row
  size_t g_tickets;   // uint32[B]  row vectors folded per sequence / tree, argmax kernel
  size_t trecs;       // TreeRec[B*(k+1)]  tree sampling: one record per node
  size_t tlist;       // uint32 count and uint32 claimed items (zero between calls), then
                      // int32[B*(k+1)] nodes with children to test
  size_t total;
};

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Rows of a sampling call: the k+1 target and k draft rows of each sequence
// (k = 0: the B rows of spec_transform_probs).
constexpr size_t sample_rows(int B, int k) { return static_cast<size_t>(B) * static_cast<size_t>(2 * k + 1); }

constexpr WsLayout ws_layout_of(size_t B, size_t rows, size_t units) {
  WsLayout w{};
  w.status = 0;
  w.s_tickets = 256;
  w.d_tickets = align_up(w.s_tickets + sizeof(uint32_t) * static_cast<size_t>(B), 256);
  w.work = align_up(w.d_tickets + sizeof(uint32_t) * static_cast<size_t>(B), 256);
  w.done = w.work + 2 * sizeof(uint32_t);
  w.hdrs = align_up(w.done + sizeof(uint32_t) * rows, 256);
  w.tags = align_up(w.hdrs + sizeof(RowHdr) * rows, 256);
  w.pubs = align_up(w.tags + sizeof(uint32_t) * kRowTags * rows, 256);
  w.csums = align_up(w.pubs + sizeof(RowPub) * rows, 256);
  w.g_slots = align_up(w.csums + sizeof(float) * kChunkRec * static_cast<size_t>(kMaxDrawChunks) * B, 256);
  w.g_tickets = align_up(w.g_slots + sizeof(uint64_t) * units, 256);
  w.trecs = align_up(w.g_tickets + sizeof(uint32_t) * static_cast<size_t>(B), 256);
  w.tlist = align_up(w.trecs + sizeof(TreeRec) * units, 256);
  w.total = align_up(w.tlist + 16 + sizeof(int32_t) * units, 256);
  return w;
}
constexpr WsLayout ws_layout(int B, int k) {
  return ws_layout_of(static_cast<size_t>(B), sample_rows(B, k), static_cast<size_t>(B) * static_cast<size_t>(k + 1));
}
// Every region grows with its count: the layout of the largest counts bounds
// the layouts of all smaller shapes.
constexpr size_t ws_bound(size_t B, size_t rows, size_t units) { return ws_layout_of(B, rows, units).total; }

struct SampleArgs {
  const void* target;          // [B][k+1][V] (MODE_PROBS: [R][V])
  const void* draft;           // [B][k][V]
  const int32_t* tokens;       // [B][k]
  const float* uniforms;       // [B][k+2]
  int B, k, V;
  float temperature;
  const float* temperature_per_seq;
  int top_k;                   // already clamped: 0 = off
  float top_p;                 // >= 1 = off
  int32_t* out_tokens;
  int32_t* out_n;
  float* out_p;
  float* out_q;
  float* out_probs;            // MODE_PROBS output [R][V]
  uint32_t* status;
  uint32_t* seq_tickets;       // [B]
  uint32_t* draw_tickets;      // [B]
  RowHdr* hdrs;                // [rows]
  uint32_t* tags;              // [rows][kRowTags]
  RowPub* pubs;                // [rows]
  float* csums;                // [B][kMaxDrawChunks][kChunkRec]
  int chunks;                  // draw chunks per sequence (<= kMaxDrawChunks)
  uint32_t* work;              // [2] fused kernel work counters
  uint32_t* done;              // [rows] fused kernel row flags
  int launch_mode;             // SPEC_LAUNCH_*
  int poll_limit;              // fused kernel: polls before a tail part gives up
  int aligned_target;          // rows start on 16-byte boundaries
  int aligned_draft;
  int mode;
  int split_grid;              // split launch: CTAs of the stream kernel
};

struct TreeSampleArgs {
  const void* logits;          // [B][N][V] target row of every node
  const void* draft;           // [B][N][V] draft row the children of every node came from
  const int32_t* tokens;       // [B][N]
  const int32_t* parents;      // [B][N]
  const float* uniforms;       // [B][N]
  int B, N, V, max_depth;
  float c;                     // log2(e) / T (scalar temperature)
  const float* temps;          // [B] per-tree temperatures, or null
  int slice;                   // elements per CTA slice (multiple of 8)
  int wchunk;                  // elements per warp chunk (multiple of 32 vectors)
  int aligned;                 // rows start on 16-byte boundaries
  int32_t* out_tokens;         // [B][max_depth+1]
  int32_t* out_path;           // [B][max_depth+1]
  int32_t* out_n;              // [B]
  uint32_t* status;
  TreeRec* recs;               // [B][N]
  uint32_t* work_count;        // nodes in work_list (zero between calls)
  uint32_t* work_next;         // node-kernel work items claimed past the first round (zero between calls)
  int32_t* work_list;          // node ids b*N + j with children to test
};

struct ArgmaxArgs {
  const void* logits;          // [B][R][V]
  const int32_t* tokens;       // chain: drafts [B][k]; tree: node tokens [B][N]
  const int32_t* parents;      // tree only
  int B, R, V;                 // R rows per sequence (k+1, or N)
  int max_depth;               // tree only
  int first_check;             // chain with R = 1: out_n = (tokens == argmax), out_tokens = argmax
  int nvr;                     // 16-byte vectors per row: ceil(V / elements per vector)
  int grid;                    // CTAs (set by the launcher)
  int aligned;
  int32_t* out_tokens;
  int32_t* out_path;
  int32_t* out_n;
  uint32_t* status;
  unsigned long long* slots;
  uint32_t* tickets;
};

struct KvArgs {
  const int32_t* path;         // [B][path_stride] or nullptr (chain)
  const int32_t* n;            // [B]
  const int32_t* base;         // [B]
  const int32_t* block_table;  // [B][max_blocks] or nullptr
  int path_stride, max_blocks, block_size, B, max_keep;
  int32_t* out_src;
  int32_t* out_dst;
  int32_t* out_new_len;
  int32_t* out_moves;          // or nullptr
  uint32_t* status;            // or nullptr
};

// Launchers (return a cudaError_t as int).  launch_sample issues the stream
// and tail kernels, and the draw kernel in MODE_SAMPLE.
int launch_sample(const SampleArgs& a, int dtype, void* stream);
int launch_argmax(const ArgmaxArgs& a, int dtype, bool tree, void* stream);
int launch_tree_sample(const TreeSampleArgs& a, int dtype, void* stream);
int launch_kv_compact(const KvArgs& a, void* stream);
// Sampling verification with one CTA per row streamed through a ring of
// bulk-copy stages: bf16 rows with or without a filter, f32 rows without one.
bool row_supported(const SampleArgs& a, int dtype);
int launch_rows(const SampleArgs& a, int dtype, void* stream);
bool split_supported(const SampleArgs& a, int dtype);
int launch_split(SampleArgs a, int dtype, void* stream);
// Shared-memory bytes of one tree-sampling CTA for slice `slice`.
size_t tree_smem_bytes(int dtype, int slice);
size_t sample_smem_bytes(int dtype, bool filter);
int num_sms();

}  // namespace specv
