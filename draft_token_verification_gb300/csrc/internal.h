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

// Per (sequence, position) result of the sampling kernel, written by the CTA
// that owns the draft token (accept, px, qx) and by the CTA that owns the
// drawn token (drawn).
struct UnitRec {
  int32_t accept;
  int32_t drawn;
  float px;
  float qx;
};

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

// What the two CTAs of a draft position (target row, draft row) hand to the
// one of them that finishes second: each row's state and probability at the
// draft token, and the target row's candidate vectors (index order), which
// hold its kept set; nlist = kPairReread when they are not listed.
constexpr int kPairList = 1024;
constexpr uint32_t kPairReread = 0xFFFFFFFFu;
struct PairRec {
  RowState rs[2];
  float xprob[2];
  uint32_t nlist;
  uint32_t pad;
  uint32_t list[kPairList];
};

// Workspace layout (byte offsets), identical for every call with the same
// (B, k).  All regions are zero between calls except the status word (the
// pair records are written before they are read).
struct WsLayout {
  size_t status;      // uint32 status word (sticky bits)
  size_t s_tickets;   // uint32[B]  arrivals per sequence, sampling kernel
  size_t s_recs;      // UnitRec[B*(k+1)]
  size_t p_tickets;   // uint32[B*k]  arrivals per draft position
  size_t p_recs;      // PairRec[B*k]
  size_t g_slots;     // uint64[B*(k+1)]  packed (value key, ~index) per row
  size_t g_tickets;   // uint32[B]  arrivals per sequence / tree, argmax kernel
  size_t total;
};

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr WsLayout ws_layout(int B, int k) {
  WsLayout w{};
  const size_t units = static_cast<size_t>(B) * static_cast<size_t>(k + 1);
  const size_t pairs = static_cast<size_t>(B) * static_cast<size_t>(k);
  w.status = 0;
  w.s_tickets = 256;
  w.s_recs = align_up(w.s_tickets + sizeof(uint32_t) * static_cast<size_t>(B), 256);
  w.p_tickets = align_up(w.s_recs + sizeof(UnitRec) * units, 256);
  w.p_recs = align_up(w.p_tickets + sizeof(uint32_t) * pairs, 256);
  w.g_slots = align_up(w.p_recs + sizeof(PairRec) * pairs, 256);
  w.g_tickets = align_up(w.g_slots + sizeof(uint64_t) * units, 256);
  w.total = align_up(w.g_tickets + sizeof(uint32_t) * static_cast<size_t>(B), 256);
  return w;
}

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
  uint32_t* tickets;
  UnitRec* recs;
  uint32_t* pair_tickets;      // [B*k]
  PairRec* pairs;              // [B*k]
  int aligned_target;          // rows start on 16-byte boundaries
  int aligned_draft;
  int mode;
};

struct ArgmaxArgs {
  const void* logits;          // [B][R][V]
  const int32_t* tokens;       // chain: drafts [B][k]; tree: node tokens [B][N]
  const int32_t* parents;      // tree only
  int B, R, V;                 // R rows per sequence (k+1, or N)
  int max_depth;               // tree only
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

// Launchers (return a cudaError_t as int).
int launch_sample(const SampleArgs& a, int dtype, int units, void* stream);
int launch_argmax(const ArgmaxArgs& a, int dtype, bool tree, void* stream);
size_t sample_smem_bytes(int dtype, bool filter);
int num_sms();

}  // namespace specv
