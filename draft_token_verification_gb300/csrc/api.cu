// api.cu -- the extern "C" boundary of libspecverify.so: argument checks on
// the host, workspace layout, launch shapes, status word and the speedup
// calculator helpers.  Declarations and the meaning of every argument are in
// include/spec_verify.h.
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "internal.h"

using namespace specv;

namespace {

std::atomic<int> g_launch_mode{SPEC_LAUNCH_AUTO};

bool dtype_ok(spec_dtype d) { return d == SPEC_F32 || d == SPEC_BF16; }
size_t elt_bytes(spec_dtype d) { return d == SPEC_BF16 ? 2 : 4; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Rows start on 16-byte boundaries: the bulk-copy / vector-load fast path.
int rows_aligned(const void* base, int V, spec_dtype d) {
  return aligned16(base) && ((static_cast<size_t>(V) * elt_bytes(d)) % 16 == 0) ? 1 : 0;
}

int check_workspace(void* ws, size_t bytes, int B, int k) {
  if (!ws) return SPEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SPEC_ERR_WORKSPACE;
  if (bytes < ws_layout(B, k).total) return SPEC_ERR_WORKSPACE;
  return SPEC_OK;
}

int run_sample(const void* target, const void* draft, const int32_t* tokens, const float* uniforms, int B, int k,
               int V, spec_dtype dtype, const spec_sampling_params* sp, int32_t* out_tokens, int32_t* out_n,
               float* out_p, float* out_q, float* out_probs, void* ws, size_t ws_bytes, void* stream, int mode,
               bool auto_split) {
  if (!dtype_ok(dtype)) return SPEC_ERR_DTYPE;
  if (!sp || !target || B < 1 || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
  if (mode == MODE_SAMPLE) {
    if (!draft || !tokens || !uniforms || !out_tokens || !out_n || k < 1 || k > SPEC_MAX_K)
      return SPEC_ERR_INVALID_ARG;
  } else if (!out_probs) {
    return SPEC_ERR_INVALID_ARG;
  }
  if (!sp->temperature_per_seq && !(sp->temperature > 0.f && isfinite(sp->temperature))) return SPEC_ERR_INVALID_ARG;
  if (sp->top_k < 0 || !(sp->top_p > 0.f && sp->top_p <= 1.f)) return SPEC_ERR_INVALID_ARG;
  const size_t es = elt_bytes(dtype);
  if (!aligned_to(target, es) || (draft && !aligned_to(draft, es)) || (tokens && !aligned_to(tokens, 4)) ||
      (uniforms && !aligned_to(uniforms, 4)))
    return SPEC_ERR_INVALID_ARG;
  const int rc = check_workspace(ws, ws_bytes, B, mode == MODE_SAMPLE ? k : 0);
  if (rc != SPEC_OK) return rc;

  SampleArgs a = {};
  a.target = target;
  a.draft = draft;
  a.tokens = tokens;
  a.uniforms = uniforms;
  a.B = B;
  a.k = mode == MODE_SAMPLE ? k : 0;
  a.V = V;
  a.temperature = sp->temperature;
  a.temperature_per_seq = sp->temperature_per_seq;
  a.top_k = (sp->top_k > 0 && sp->top_k < V) ? sp->top_k : 0;
  a.top_p = sp->top_p;
  a.out_tokens = out_tokens;
  a.out_n = out_n;
  a.out_p = out_p;
  a.out_q = out_q;
  a.out_probs = out_probs;
  const WsLayout L = ws_layout(B, a.k);
  unsigned char* w = static_cast<unsigned char*>(ws);
  a.status = reinterpret_cast<uint32_t*>(w + L.status);
  a.seq_tickets = reinterpret_cast<uint32_t*>(w + L.s_tickets);
  a.draw_tickets = reinterpret_cast<uint32_t*>(w + L.d_tickets);
  a.hdrs = reinterpret_cast<RowHdr*>(w + L.hdrs);
  a.tags = reinterpret_cast<uint32_t*>(w + L.tags);
  a.pubs = reinterpret_cast<RowPub*>(w + L.pubs);
  a.csums = reinterpret_cast<float*>(w + L.csums);
  a.work = reinterpret_cast<uint32_t*>(w + L.work);
  a.launch_mode = g_launch_mode.load();
  if (a.launch_mode == SPEC_LAUNCH_AUTO) {
    // the split launch where the nucleus reaches deep below the row maximum
    // (top-p >= 0.95) or the temperature varies per sequence; else fused
    const bool deep = a.top_p >= 0.95f && a.top_p < 1.f;
    a.launch_mode = (auto_split && (deep || a.temperature_per_seq)) ? SPEC_LAUNCH_SPLIT : SPEC_LAUNCH_FUSED;
  }
  a.done = reinterpret_cast<uint32_t*>(w + L.done);
  // the draw at the first rejection: a few chunks over listed vectors, more
  // over whole rows (no filter)
  a.chunks = (a.top_k > 0 || a.top_p < 1.f) ? 8 : kMaxDrawChunks;
  a.aligned_target = rows_aligned(target, V, dtype);
  a.aligned_draft = draft ? rows_aligned(draft, V, dtype) : 0;
  a.mode = mode;
  const int dt = dtype == SPEC_BF16 ? DT_BF16 : DT_F32;
  if (a.launch_mode == SPEC_LAUNCH_SPLIT) {
    if (split_supported(a, dt)) {
      const int e = launch_split(a, dt, stream);
      if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return SPEC_ERR_LAUNCH;
      return SPEC_OK;
    }
    a.launch_mode = SPEC_LAUNCH_FUSED;
  }
  const bool rows = a.launch_mode == SPEC_LAUNCH_ROWS || a.launch_mode == SPEC_LAUNCH_FUSED_WAIT_TEST;
  if (rows && row_supported(a, dt)) {
    a.poll_limit = 64;  // (used only by the failure-detection mode)
    const int e = launch_rows(a, dt, stream);
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return SPEC_ERR_LAUNCH;
    return SPEC_OK;
  }
  if (a.launch_mode == SPEC_LAUNCH_ROWS) a.launch_mode = SPEC_LAUNCH_FUSED;
  const int e = launch_sample(a, dt, stream);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return SPEC_ERR_LAUNCH;
  return SPEC_OK;
}

// Elements of one 16-byte vector.
int vec_elems(spec_dtype d) { return 16 / static_cast<int>(elt_bytes(d)); }

// ------------------------------------------------ allocation-free sampling
// Fixed scratch for spec_verify_sample_noalloc: a bound on the workspace
// layout of every shape it accepts (B <= SPEC_NOALLOC_MAX_B and B*(k+1) <=
// SPEC_NOALLOC_MAX_UNITS, so at most 2 * SPEC_NOALLOC_MAX_UNITS rows).  Every
// GPU that loads the library holds one copy until the process exits.
constexpr size_t kNoAllocBytes = ws_bound(SPEC_NOALLOC_MAX_B, 2 * static_cast<size_t>(SPEC_NOALLOC_MAX_UNITS),
                                          SPEC_NOALLOC_MAX_UNITS);
constexpr int kNoAllocMaxDevices = 64;

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

}  // namespace

// In host code this name stands for the array only as a handle for the
// runtime; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (with that device current) and cached.
int noalloc_scratch(unsigned char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_LAUNCH;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return SPEC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPEC_ERR_LAUNCH;
    g_noalloc_ptr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_noalloc_ptr[dev]);
  return SPEC_OK;
}

}  // namespace

extern "C" {

size_t spec_verify_workspace_size(int B, int k, int V, spec_dtype dtype) {
  if (B < 1 || k < 0 || k > SPEC_MAX_TREE_NODES || V < 1 || V > SPEC_MAX_V || !dtype_ok(dtype)) return 0;
  return ws_layout(B, k).total;
}

int spec_verify_sample(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                       const float* uniforms, int B, int k, int V, spec_dtype dtype,
                       const spec_sampling_params* params, int32_t* out_tokens, int32_t* out_num_accepted,
                       float* out_p_draft, float* out_q_draft, void* workspace, size_t workspace_bytes,
                       void* cuda_stream) {
  return run_sample(target_logits, draft_logits, draft_tokens, uniforms, B, k, V, dtype, params, out_tokens,
                    out_num_accepted, out_p_draft, out_q_draft, nullptr, workspace, workspace_bytes, cuda_stream,
                    MODE_SAMPLE, true);
}

int spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                               const float* uniforms, int B, int k, int V, spec_dtype dtype,
                               const spec_sampling_params* params, int32_t* out_tokens, int32_t* out_num_accepted,
                               float* out_p_draft, float* out_q_draft, uint32_t* out_status, void* cuda_stream) {
  if (B < 1 || k < 1 || k > SPEC_MAX_K) return SPEC_ERR_INVALID_ARG;
  if (B > SPEC_NOALLOC_MAX_B || static_cast<long long>(B) * (k + 1) > SPEC_NOALLOC_MAX_UNITS)
    return SPEC_ERR_SCRATCH_LIMIT;
  const WsLayout L = ws_layout(B, k);
  if (L.total > kNoAllocBytes) return SPEC_ERR_SCRATCH_LIMIT;
  if (out_status && !aligned_to(out_status, sizeof(uint32_t))) return SPEC_ERR_INVALID_ARG;
  unsigned char* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != SPEC_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  // The array keeps whatever the previous call left: the status word and the
  // tickets must start at zero (everything else is written before it is read).
  if (cudaMemsetAsync(scratch, 0, L.hdrs, st) != cudaSuccess) return SPEC_ERR_LAUNCH;
  rc = run_sample(target_logits, draft_logits, draft_tokens, uniforms, B, k, V, dtype, params, out_tokens,
                  out_num_accepted, out_p_draft, out_q_draft, nullptr, scratch, kNoAllocBytes, cuda_stream,
                  MODE_SAMPLE, false);
  if (rc != SPEC_OK) return rc;
  if (out_status && cudaMemcpyAsync(out_status, scratch + L.status, sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                                    st) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return SPEC_OK;
}

int spec_sample_launch_mode(int mode) {
  if (mode != SPEC_LAUNCH_FUSED && mode != SPEC_LAUNCH_SEPARATE && mode != SPEC_LAUNCH_FUSED_WAIT_TEST &&
      mode != SPEC_LAUNCH_ROWS && mode != SPEC_LAUNCH_SPLIT && mode != SPEC_LAUNCH_AUTO)
    return SPEC_ERR_INVALID_ARG;
  return g_launch_mode.exchange(mode);
}

int spec_kv_compact(const int32_t* path, int path_stride, const int32_t* num_accepted, const int32_t* kv_base,
                    const int32_t* block_table, int max_blocks, int block_size, int B, int max_keep,
                    int32_t* out_src, int32_t* out_dst, int32_t* out_new_len, int32_t* out_num_moves,
                    uint32_t* out_status, void* cuda_stream) {
  if (!num_accepted || !kv_base || !out_src || !out_dst || !out_new_len) return SPEC_ERR_INVALID_ARG;
  if (B < 1 || max_keep < 1) return SPEC_ERR_INVALID_ARG;
  if (path && path_stride < 1) return SPEC_ERR_INVALID_ARG;
  if (block_table && (block_size < 1 || max_blocks < 1)) return SPEC_ERR_INVALID_ARG;
  const void* ptrs[] = {path, num_accepted, kv_base, block_table, out_src, out_dst, out_new_len, out_num_moves,
                        out_status};
  for (const void* q : ptrs)
    if (q && !aligned_to(q, 4)) return SPEC_ERR_INVALID_ARG;
  KvArgs a = {};
  a.path = path;
  a.n = num_accepted;
  a.base = kv_base;
  a.block_table = block_table;
  a.path_stride = path ? path_stride : 0;
  a.max_blocks = block_table ? max_blocks : 0;
  a.block_size = block_table ? block_size : 0;
  a.B = B;
  a.max_keep = max_keep;
  a.out_src = out_src;
  a.out_dst = out_dst;
  a.out_new_len = out_new_len;
  a.out_moves = out_num_moves;
  a.status = out_status;
  if (launch_kv_compact(a, cuda_stream) != cudaSuccess) return SPEC_ERR_LAUNCH;
  return SPEC_OK;
}

int spec_transform_probs(const void* logits, int R, int V, spec_dtype dtype, const spec_sampling_params* params,
                         float* out_probs, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  return run_sample(logits, nullptr, nullptr, nullptr, R, 0, V, dtype, params, nullptr, nullptr, nullptr, nullptr,
                    out_probs, workspace, workspace_bytes, cuda_stream, MODE_PROBS, false);
}

int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B, int k, int V,
                       spec_dtype dtype, int32_t* out_tokens, int32_t* out_num_accepted, void* workspace,
                       size_t workspace_bytes, void* cuda_stream) {
  if (!dtype_ok(dtype)) return SPEC_ERR_DTYPE;
  if (!target_logits || !draft_tokens || !out_tokens || !out_num_accepted) return SPEC_ERR_INVALID_ARG;
  if (B < 1 || k < 1 || k > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
  if (!aligned_to(target_logits, elt_bytes(dtype)) || !aligned_to(draft_tokens, 4)) return SPEC_ERR_INVALID_ARG;
  const int rc = check_workspace(workspace, workspace_bytes, B, k);
  if (rc != SPEC_OK) return rc;
  const WsLayout L = ws_layout(B, k);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  ArgmaxArgs a = {};
  a.logits = target_logits;
  a.tokens = draft_tokens;
  a.B = B;
  a.R = k + 1;
  a.V = V;
  a.nvr = (V + vec_elems(dtype) - 1) / vec_elems(dtype);
  a.aligned = rows_aligned(target_logits, V, dtype);
  a.out_tokens = out_tokens;
  a.out_n = out_num_accepted;
  a.status = reinterpret_cast<uint32_t*>(w + L.status);
  a.slots = reinterpret_cast<unsigned long long*>(w + L.g_slots);
  a.tickets = reinterpret_cast<uint32_t*>(w + L.g_tickets);
  if (launch_argmax(a, dtype == SPEC_BF16 ? DT_BF16 : DT_F32, false, cuda_stream) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return SPEC_OK;
}

int spec_first_draft_check(const void* prev_rows, const int32_t* draft0, int B, int V, spec_dtype dtype,
                           int32_t* out_accept, int32_t* out_argmax, void* workspace, size_t workspace_bytes,
                           void* cuda_stream) {
  if (!dtype_ok(dtype)) return SPEC_ERR_DTYPE;
  if (!prev_rows || !draft0 || !out_accept || !out_argmax) return SPEC_ERR_INVALID_ARG;
  if (B < 1 || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
  if (!aligned_to(prev_rows, elt_bytes(dtype)) || !aligned_to(draft0, 4)) return SPEC_ERR_INVALID_ARG;
  const int rc = check_workspace(workspace, workspace_bytes, B, 1);
  if (rc != SPEC_OK) return rc;
  const WsLayout L = ws_layout(B, 1);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  ArgmaxArgs a = {};
  a.logits = prev_rows;
  a.tokens = draft0;
  a.B = B;
  a.R = 1;
  a.V = V;
  a.first_check = 1;
  a.nvr = (V + vec_elems(dtype) - 1) / vec_elems(dtype);
  a.aligned = rows_aligned(prev_rows, V, dtype);
  a.out_tokens = out_argmax;
  a.out_n = out_accept;
  a.status = reinterpret_cast<uint32_t*>(w + L.status);
  a.slots = reinterpret_cast<unsigned long long*>(w + L.g_slots);
  a.tickets = reinterpret_cast<uint32_t*>(w + L.g_tickets);
  if (launch_argmax(a, dtype == SPEC_BF16 ? DT_BF16 : DT_F32, false, cuda_stream) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return SPEC_OK;
}

// The tree kernels stage one tree's parents, tokens and outcomes in shared
// arrays of kMaxTreeNodes entries; the largest N the entry points accept fits.
static_assert(SPEC_MAX_TREE_NODES <= kMaxTreeNodes, "a tree of SPEC_MAX_TREE_NODES nodes must fit the tree kernels");

int spec_verify_tree_greedy(const void* node_logits, const int32_t* node_tokens, const int32_t* parents, int B,
                            int N, int V, int max_depth, spec_dtype dtype, int32_t* out_tokens, int32_t* out_path,
                            int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                            void* cuda_stream) {
  if (!dtype_ok(dtype)) return SPEC_ERR_DTYPE;
  if (!node_logits || !node_tokens || !parents || !out_tokens || !out_path || !out_num_accepted)
    return SPEC_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || N > SPEC_MAX_TREE_NODES || V < 1 || V > SPEC_MAX_V || max_depth < 1)
    return SPEC_ERR_INVALID_ARG;
  if (!aligned_to(node_logits, elt_bytes(dtype)) || !aligned_to(node_tokens, 4) || !aligned_to(parents, 4))
    return SPEC_ERR_INVALID_ARG;
  const int rc = check_workspace(workspace, workspace_bytes, B, N - 1);
  if (rc != SPEC_OK) return rc;
  const WsLayout L = ws_layout(B, N - 1);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  ArgmaxArgs a = {};
  a.logits = node_logits;
  a.tokens = node_tokens;
  a.parents = parents;
  a.B = B;
  a.R = N;
  a.V = V;
  a.max_depth = max_depth;
  a.nvr = (V + vec_elems(dtype) - 1) / vec_elems(dtype);
  a.aligned = rows_aligned(node_logits, V, dtype);
  a.out_tokens = out_tokens;
  a.out_path = out_path;
  a.out_n = out_num_accepted;
  a.status = reinterpret_cast<uint32_t*>(w + L.status);
  a.slots = reinterpret_cast<unsigned long long*>(w + L.g_slots);
  a.tickets = reinterpret_cast<uint32_t*>(w + L.g_tickets);
  if (launch_argmax(a, dtype == SPEC_BF16 ? DT_BF16 : DT_F32, true, cuda_stream) != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return SPEC_OK;
}

int spec_verify_tree_sample(const void* node_logits, const void* draft_logits, const int32_t* node_tokens,
                            const int32_t* parents, const float* uniforms, int B, int N, int V, int max_depth,
                            spec_dtype dtype, float temperature, const float* temperature_per_tree,
                            int32_t* out_tokens, int32_t* out_path,
                            int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                            void* cuda_stream) {
  if (!dtype_ok(dtype)) return SPEC_ERR_DTYPE;
  if (!node_logits || !draft_logits || !node_tokens || !parents || !uniforms || !out_tokens || !out_path ||
      !out_num_accepted)
    return SPEC_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || N > SPEC_MAX_TREE_NODES || V < 1 || V > SPEC_MAX_V || max_depth < 1)
    return SPEC_ERR_INVALID_ARG;
  if (!temperature_per_tree && !(temperature > 0.f && isfinite(temperature))) return SPEC_ERR_INVALID_ARG;
  const size_t es = elt_bytes(dtype);
  if (!aligned_to(node_logits, es) || !aligned_to(draft_logits, es) || !aligned_to(node_tokens, 4) ||
      !aligned_to(parents, 4) || !aligned_to(uniforms, 4) ||
      (temperature_per_tree && !aligned_to(temperature_per_tree, 4)))
    return SPEC_ERR_INVALID_ARG;
  const int rc = check_workspace(workspace, workspace_bytes, B, N - 1);
  if (rc != SPEC_OK) return rc;
  // each CTA of a node's cluster holds 1/kTreeCl of both rows in shared memory
  const int slice = ((V + kTreeCl - 1) / kTreeCl + 7) / 8 * 8;
  if (tree_smem_bytes(dtype == SPEC_BF16 ? DT_BF16 : DT_F32, slice) > kTreeSmemMax) return SPEC_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(B, N - 1);
  unsigned char* w = static_cast<unsigned char*>(workspace);
  TreeSampleArgs a = {};
  a.logits = node_logits;
  a.draft = draft_logits;
  a.tokens = node_tokens;
  a.parents = parents;
  a.uniforms = uniforms;
  a.B = B;
  a.N = N;
  a.V = V;
  a.max_depth = max_depth;
  a.c = temperature_per_tree ? 0.f : 1.4426950408889634f / temperature;  // log2(e) / T, as in the chain kernels
  a.temps = temperature_per_tree;
  a.slice = slice;
  // warp chunks are whole rounds of 32 lanes x one 16-byte vector
  const int round_elems = 32 * vec_elems(dtype);
  a.wchunk = ((slice + kWarps - 1) / kWarps + round_elems - 1) / round_elems * round_elems;
  a.aligned = rows_aligned(node_logits, V, dtype) && rows_aligned(draft_logits, V, dtype);
  a.out_tokens = out_tokens;
  a.out_path = out_path;
  a.out_n = out_num_accepted;
  a.status = reinterpret_cast<uint32_t*>(w + L.status);
  a.recs = reinterpret_cast<TreeRec*>(w + L.trecs);
  a.work_count = reinterpret_cast<uint32_t*>(w + L.tlist);
  a.work_next = reinterpret_cast<uint32_t*>(w + L.tlist + 4);
  a.work_list = reinterpret_cast<int32_t*>(w + L.tlist + 16);
  if (launch_tree_sample(a, dtype == SPEC_BF16 ? DT_BF16 : DT_F32, cuda_stream) != cudaSuccess ||
      cudaGetLastError() != cudaSuccess)
    return SPEC_ERR_LAUNCH;
  return SPEC_OK;
}

int spec_get_status(void* workspace, uint32_t* status, void* cuda_stream) {
  if (!workspace || !status) return SPEC_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  uint32_t* dev = static_cast<uint32_t*>(workspace);
  uint32_t host = 0;
  if (cudaMemcpyAsync(&host, dev, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess) return SPEC_ERR_LAUNCH;
  if (cudaMemsetAsync(dev, 0, sizeof(uint32_t), st) != cudaSuccess) return SPEC_ERR_LAUNCH;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SPEC_ERR_LAUNCH;
  *status = host;
  if (host & SPEC_STATUS_TIMEOUT) return SPEC_ERR_TIMEOUT;
  return host ? SPEC_ERR_DEVICE_DATA : SPEC_OK;
}

const char* spec_error_string(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_DTYPE: return "unsupported dtype";
    case SPEC_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case SPEC_ERR_LAUNCH: return "CUDA launch or copy failed";
    case SPEC_ERR_DEVICE_DATA: return "device found invalid data (see status bits)";
    case SPEC_ERR_TIMEOUT: return "a bounded device wait gave up";
    case SPEC_ERR_UNSUPPORTED: return "shape beyond the library's limits";
    case SPEC_ERR_SCRATCH_LIMIT:
      return "B > 256 or B*(k+1) > 256: beyond the fixed scratch of spec_verify_sample_noalloc";
    default: return "unknown error code";
  }
}

double spec_expected_tokens(double alpha, int gamma) {
  double e = 0.0, p = 1.0;
  for (int i = 0; i <= gamma; ++i) {
    e += p;
    p *= alpha;
  }
  return e;
}

double spec_improvement_factor(double alpha, int gamma, double c) {
  return spec_expected_tokens(alpha, gamma) / (static_cast<double>(gamma) * c + 1.0);
}

double spec_break_even_acceptance(int k) { return static_cast<double>(k) / static_cast<double>(k + 1); }

int spec_best_gamma(double alpha, double c, int gamma_max, double* best_factor) {
  if (!(alpha >= 0.0 && alpha <= 1.0) || !(c >= 0.0) || gamma_max < 1 || gamma_max > 64) return SPEC_ERR_INVALID_ARG;
  int arg = 1;
  double top = spec_improvement_factor(alpha, 1, c);
  for (int g = 2; g <= gamma_max; ++g) {
    const double f = spec_improvement_factor(alpha, g, c);
    if (f > top) {
      top = f;
      arg = g;
    }
  }
  if (best_factor) *best_factor = top;
  return arg;
}

}  // extern "C"
