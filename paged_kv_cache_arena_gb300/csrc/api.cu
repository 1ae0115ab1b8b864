// C ABI of the library (declared in include/kshipra.h): argument validation,
// options, the device status word, TMA descriptors and kernel dispatch.
//
// Pages "Building Kshipra" part 3 (kshipra-3): the arena is reserved once by
// the caller and never reallocated here (section 1); attention reads it in
// place through block tables (section 4); a call may mix prefill chunks with
// decodes (section 5).  Host-side checks run before anything is enqueued.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

using namespace kshipra;

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(KSHIPRA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Tuning options (kshipra_set_option), one set per host thread: a thread's
// calls and its workspace queries see only its own settings, so threads (or
// libraries) that tune differently never change each other's kernels or
// workspace sizes.
thread_local int g_opt_split_tokens = 0;
thread_local int g_opt_decode_max_rows = kDecodeMaxRows;

// A mixed batch (decode-class and prefill-class rows, head_dim 128) runs its
// prefill kernel on a side stream of the calling thread, beside the decode
// kernel: a fork event on the caller's stream, the pair kernel on the side
// stream (highest priority, so that its clusters are placed before the
// decode CTAs fill the SMs), the decode kernel on the caller's stream, and a
// join event the caller's stream waits for.  Created on first use, one set
// per (thread, device); released when the thread ends.  Callers that must not
// create anything (the no-alloc entry point) turn it off for their call.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  int device = -1;
  ~SideStream() {
    if (join) cudaEventDestroy(join);
    if (fork) cudaEventDestroy(fork);
    if (stream) cudaStreamDestroy(stream);
  }
};
thread_local SideStream g_side[8];
thread_local bool g_side_off = false;

// The calling thread's side stream on the current device, or null (none
// could be made, the device index is past the table, or side streams are off).
SideStream* side_stream() {
  if (g_side_off) return nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 8) {
    cudaGetLastError();
    return nullptr;
  }
  SideStream& ss = g_side[dev];
  if (ss.device == dev) return &ss;
  int least = 0, greatest = 0;
  if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
      cudaStreamCreateWithPriority(&ss.stream, cudaStreamNonBlocking, greatest) != cudaSuccess ||
      cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;  // the destructor releases whatever was made
  }
  ss.device = dev;
  return &ss;
}

// ---- device status word ------------------------------------------------
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
unsigned* g_status_ptr[kMaxDevices] = {};

cudaError_t status_ptr(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

// The SM count of the current device.  The first call on a host thread (and
// after a change of device) also makes the device's primary context current
// there: the driver-API tensor-map encoder needs one, and a thread whose CUDA
// work went through other libraries so far may have none bound yet.
cudaError_t sm_count_current(int* out) {
  thread_local int bound = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (bound != dev) {
    if ((e = cudaSetDevice(dev)) != cudaSuccess) return e;
    bound = dev;
  }
  return cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
}

// ---- TMA descriptors -----------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return g_encode;
}

// 2-D view of an arena: rows (block, kv head, slot), columns head_dim; boxes
// of box_rows x 64 elements with the 128-byte swizzle.
int arena_map(CUtensorMap* map, const void* arena, int dtype, int head_dim, long long rows, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return fail(KSHIPRA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dtype == KSHIPRA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   2, const_cast<void*>(arena), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KSHIPRA_ERR_CUDA, "cuTensorMapEncodeTiled(arena) failed (%d)", (int)r);
  return KSHIPRA_OK;
}

// 3-D view of q_rot [tokens][q heads][head_dim]; one box = `tokens` tokens x
// `group` heads x 64 columns, i.e. the 128 rows (token, head-in-group) of a
// prefill tile.
int query_map(CUtensorMap* map, const void* q, int dtype, int head_dim, int num_q_heads, int num_tokens,
              int group) {
  auto enc = encode_fn();
  if (!enc) return fail(KSHIPRA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_q_heads),
                        static_cast<cuuint64_t>(num_tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                           static_cast<cuuint64_t>(head_dim) * 2 * num_q_heads};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(128 / group)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dtype == KSHIPRA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   3, const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KSHIPRA_ERR_CUDA, "cuTensorMapEncodeTiled(q) failed (%d)", (int)r);
  return KSHIPRA_OK;
}

// ---- shape checks ----------------------------------------------------------
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_heads(int num_q_heads, int num_kv_heads, int head_dim, int block_size, int dtype) {
  if (num_q_heads <= 0 || num_kv_heads <= 0)
    return fail(KSHIPRA_ERR_INVALID_ARG, "head counts must be positive (q %d, kv %d)", num_q_heads, num_kv_heads);
  if (num_q_heads % num_kv_heads)
    return fail(KSHIPRA_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                num_kv_heads);
  const int g = num_q_heads / num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16)
    return fail(KSHIPRA_ERR_UNSUPPORTED, "group size %d not in {1, 2, 4, 8, 16}", g);
  if (num_kv_heads > 255) return fail(KSHIPRA_ERR_UNSUPPORTED, "num_kv_heads %d above 255", num_kv_heads);
  if (head_dim != 64 && head_dim != 128) return fail(KSHIPRA_ERR_UNSUPPORTED, "head_dim %d not in {64, 128}", head_dim);
  if (block_size != 16 && block_size != 32)
    return fail(KSHIPRA_ERR_UNSUPPORTED, "block_size %d not in {16, 32}", block_size);
  if (dtype != KSHIPRA_DTYPE_F16 && dtype != KSHIPRA_DTYPE_BF16)
    return fail(KSHIPRA_ERR_UNSUPPORTED, "dtype %d not in {0 (f16), 1 (bf16)}", dtype);
  return KSHIPRA_OK;
}

int check_arena(int num_blocks, int num_kv_heads, int block_size, int max_blocks_per_seq) {
  if (num_blocks <= 0 || max_blocks_per_seq <= 0)
    return fail(KSHIPRA_ERR_INVALID_ARG, "num_blocks %d and max_blocks_per_seq %d must be positive", num_blocks,
                max_blocks_per_seq);
  if (static_cast<long long>(num_blocks) * num_kv_heads * block_size >= (1ll << 31))
    return fail(KSHIPRA_ERR_UNSUPPORTED, "arena rows (num_blocks x kv heads x block_size) must stay below 2^31");
  if (static_cast<long long>(max_blocks_per_seq) * block_size >= (1ll << 30))
    return fail(KSHIPRA_ERR_UNSUPPORTED, "max_blocks_per_seq x block_size must stay below 2^30");
  return KSHIPRA_OK;
}

// Keys per decode split.  Aims at about kDecodeWaves wave of two CTAs per SM
// for the largest batch these arguments allow, in multiples of 64 keys
// between 256 and kDecodeMaxSplit.  The decode kernel starts its CTAs longest
// first, so the last wave holds the shortest work and few long splits beat
// many short ones: every split pays its own start (a pipeline fill, the unit
// lookup) and, when a sequence has several, a partial write and a merge.  On
// GB300 (one wave, 8 K cap) a 64 x 8 head batch at contexts up to 4096 runs one
// CTA per (sequence, kv head) at 0.88 of the copy bandwidth, against 0.81 at
// two waves, 0.73 at three and 0.77 for the earlier in-order grid at four; 16
// sequences of 32 K keys run at the copy bandwidth with four 8 K splits.
constexpr int kDecodeWaves = 1;
constexpr int kDecodeMaxSplit = 8192;

int split_tokens_for(int num_seqs, int max_context_len, int num_kv_heads, int sm_count) {
  const int opt = g_opt_split_tokens;
  if (opt > 0) return opt;
  const long long units = static_cast<long long>(num_seqs) * num_kv_heads;
  const long long target = static_cast<long long>(kDecodeWaves) * 2 * (sm_count > 0 ? sm_count : 1);
  long long L = (static_cast<long long>(max_context_len) * units + target - 1) / target;
  L = (L + 63) / 64 * 64;
  if (L < 256) L = 256;
  if (L > kDecodeMaxSplit) L = kDecodeMaxSplit;
  const long long cap = (static_cast<long long>(max_context_len) + 63) / 64 * 64;
  if (L > cap) L = cap < 64 ? 64 : cap;
  return static_cast<int>(L);
}

struct WorkspacePlan {
  int split_tokens;
  int max_splits;
  int max_items;
  size_t o_bytes, ml_bytes, counter_bytes, items_bytes, total;
};

WorkspacePlan plan_workspace(int num_seqs, int num_tokens, int max_context_len, int num_q_heads,
                             int num_kv_heads, int head_dim, int sm_count) {
  WorkspacePlan p{};
  auto round256 = [](size_t x) { return (x + 255) / 256 * 256; };
  p.split_tokens = split_tokens_for(num_seqs, max_context_len, num_kv_heads, sm_count);
  p.max_splits = max_context_len > 0 ? (max_context_len + p.split_tokens - 1) / p.split_tokens : 1;
  if (p.max_splits < 1) p.max_splits = 1;
  if (p.max_splits > 1 && g_opt_decode_max_rows > 0) {  // decode partials and counters
    const size_t rows = static_cast<size_t>(p.max_splits) * num_tokens * num_q_heads;
    p.o_bytes = round256(rows * head_dim * sizeof(float));
    p.ml_bytes = round256(rows * 2 * sizeof(float));
    p.counter_bytes = round256(static_cast<size_t>(num_seqs) * num_kv_heads * sizeof(unsigned));
  }
  // prefill work list + its length
  p.max_items = num_tokens > 0 ? prefill_max_items(num_seqs, num_tokens, num_q_heads, num_kv_heads) : 0;
  p.items_bytes = p.max_items > 0 ? round256(static_cast<size_t>(p.max_items) * sizeof(uint64_t) + sizeof(int)) : 0;
  p.total = p.o_bytes + p.ml_bytes + p.counter_bytes + p.items_bytes;
  return p;
}

// Host checks of kshipra_kv_append_rope and its launch arguments.
int append_prepare(AppendArgs* out, const void* q, const void* k, const void* v, void* q_rot, void* k_arena,
                   void* v_arena, const int32_t* block_tables, const int32_t* query_start_loc,
                   const int32_t* positions, const float* rope_table, int rope_max_pos, int num_seqs, int num_tokens,
                   int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                   int num_blocks, int dtype) {
  if (num_seqs < 0 || num_tokens < 0) return fail(KSHIPRA_ERR_INVALID_ARG, "negative num_seqs or num_tokens");
  if (num_seqs == 0 && num_tokens > 0) return fail(KSHIPRA_ERR_INVALID_ARG, "tokens without sequences");
  int rc = check_heads(num_q_heads, num_kv_heads, head_dim, block_size, dtype);
  if (rc) return rc;
  if ((rc = check_arena(num_blocks, num_kv_heads, block_size, max_blocks_per_seq))) return rc;
  if ((q == nullptr) != (q_rot == nullptr))
    return fail(KSHIPRA_ERR_INVALID_ARG, "q and q_rot must both be given or both be NULL");
  if (rope_max_pos <= 0) return fail(KSHIPRA_ERR_INVALID_ARG, "rope_max_pos must be positive");
  if (num_tokens == 0) return KSHIPRA_OK;
  if (!k || !v || !k_arena || !v_arena || !block_tables || !query_start_loc || !positions || !rope_table)
    return fail(KSHIPRA_ERR_INVALID_ARG, "a required pointer is NULL");
  const void* vec[] = {q, k, v, q_rot, k_arena, v_arena, rope_table};
  for (const void* p : vec)
    if (p && !aligned(p, 16)) return fail(KSHIPRA_ERR_INVALID_ARG, "data pointers must be 16-byte aligned");
  AppendArgs& a = *out;
  a.q = q; a.k = k; a.v = v; a.q_rot = q_rot; a.k_arena = k_arena; a.v_arena = v_arena;
  a.block_tables = block_tables; a.query_start_loc = query_start_loc; a.positions = positions;
  a.rope_table = rope_table; a.rope_max_pos = rope_max_pos;
  a.num_seqs = num_seqs; a.num_tokens = num_tokens; a.num_q_heads = num_q_heads; a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim; a.block_size = block_size; a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks; a.dtype = dtype;
  cudaError_t e = status_ptr(&a.status);
  if (e != cudaSuccess) return cuda_fail(e, "status word");
  if ((e = sm_count_current(&a.sm_count)) != cudaSuccess) return cuda_fail(e, "SM count");
  return KSHIPRA_OK;
}

// The new tokens' raw rows for the fused step (see AttnArgs): k and v NULL
// when a separate append writes them (the kernels then only rotate q).
struct FusedInputs {
  const void* q;
  const void* k;
  const void* v;
  const float* rope_table;
  int rope_max_pos;
  void* q_rot_out;
  void* k_arena;
  void* v_arena;
};

// kshipra_paged_attention, or with fz a fused step (q_rot then is an optional
// output): every sequence of the decode class with fz->k set (one launch that
// also appends), or, with fz->k NULL, attention kernels that rotate q after a
// separate K/V append, launched as its programmatic dependents (dependent).
// validate_only: return after the host-side checks, before any CUDA work.
int attention_impl(void* out, const void* q_rot, const void* k_arena, const void* v_arena,
                   const int32_t* block_tables, const int32_t* context_lens, const int32_t* query_start_loc,
                   const int32_t* positions, int num_seqs, int num_tokens, int max_query_len, int max_context_len,
                   int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                   int num_blocks, float scale, int dtype, void* workspace, size_t workspace_bytes, void* stream,
                   const FusedInputs* fz, bool dependent = false, bool validate_only = false) {
  if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0 || max_context_len < 0)
    return fail(KSHIPRA_ERR_INVALID_ARG, "negative size argument");
  if (num_seqs == 0 && num_tokens > 0) return fail(KSHIPRA_ERR_INVALID_ARG, "tokens without sequences");
  int rc = check_heads(num_q_heads, num_kv_heads, head_dim, block_size, dtype);
  if (rc) return rc;
  if ((rc = check_arena(num_blocks, num_kv_heads, block_size, max_blocks_per_seq))) return rc;
  if (num_seqs >= (1 << 24) || max_query_len / (2 * (128 / (num_q_heads / num_kv_heads))) >= (1 << 16))
    return fail(KSHIPRA_ERR_UNSUPPORTED, "num_seqs must stay below 2^24 and max_query_len below 2^16 tile pairs");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(KSHIPRA_ERR_INVALID_ARG, "scale must be positive");
  if (num_tokens == 0) return KSHIPRA_OK;
  if (max_context_len <= 0 || max_query_len <= 0)
    return fail(KSHIPRA_ERR_INVALID_ARG, "max_context_len and max_query_len must be positive");
  if (static_cast<long long>(max_context_len) > static_cast<long long>(max_blocks_per_seq) * block_size)
    return fail(KSHIPRA_ERR_INVALID_ARG, "max_context_len %d exceeds max_blocks_per_seq x block_size",
                max_context_len);
  if (!out || (!q_rot && !fz) || !k_arena || !v_arena || !block_tables || !context_lens || !query_start_loc ||
      !positions)
    return fail(KSHIPRA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (out == q_rot) return fail(KSHIPRA_ERR_INVALID_ARG, "out must not alias q_rot");
  const void* vec[] = {out, q_rot, k_arena, v_arena};
  for (const void* p : vec)
    if (p && !aligned(p, 16)) return fail(KSHIPRA_ERR_INVALID_ARG, "data pointers must be 16-byte aligned");
  int sms = 0;
  cudaError_t e = sm_count_current(&sms);
  if (e != cudaSuccess) return cuda_fail(e, "SM count");
  const WorkspacePlan plan =
      plan_workspace(num_seqs, num_tokens, max_context_len, num_q_heads, num_kv_heads, head_dim, sms);
  if (workspace_bytes < plan.total)
    return fail(KSHIPRA_ERR_WORKSPACE_TOO_SMALL, "workspace of %zu bytes, %zu needed", workspace_bytes, plan.total);
  if (plan.total && (!workspace || !aligned(workspace, 256)))
    return fail(KSHIPRA_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
  if (validate_only) return KSHIPRA_OK;

  AttnArgs a{};
  a.out = out; a.q_rot = q_rot; a.block_tables = block_tables; a.context_lens = context_lens;
  a.query_start_loc = query_start_loc; a.positions = positions;
  char* ws = static_cast<char*>(workspace);
  a.ws_o = plan.o_bytes ? reinterpret_cast<float*>(ws) : nullptr;
  a.ws_ml = plan.ml_bytes ? reinterpret_cast<float*>(ws + plan.o_bytes) : nullptr;
  a.ws_counters = plan.counter_bytes ? reinterpret_cast<unsigned*>(ws + plan.o_bytes + plan.ml_bytes) : nullptr;
  const size_t items_off = plan.o_bytes + plan.ml_bytes + plan.counter_bytes;
  a.ws_items = plan.items_bytes ? reinterpret_cast<uint64_t*>(ws + items_off) : nullptr;
  a.ws_item_count =
      plan.items_bytes ? reinterpret_cast<int*>(ws + items_off + static_cast<size_t>(plan.max_items) * 8) : nullptr;
  a.max_items = plan.max_items;
  a.sm_count = sms;
  a.num_seqs = num_seqs; a.num_tokens = num_tokens; a.max_query_len = max_query_len;
  a.max_context_len = max_context_len; a.num_q_heads = num_q_heads; a.num_kv_heads = num_kv_heads;
  a.group = num_q_heads / num_kv_heads; a.head_dim = head_dim; a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq; a.num_blocks = num_blocks;
  a.split_tokens = plan.split_tokens; a.max_splits = plan.max_splits;
  a.decode_max_rows = g_opt_decode_max_rows;
  a.decode_ordered = num_seqs <= kDecodeOrderedMaxSeqs ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.dtype = dtype;
  if (fz) {
    a.q_raw = fz->q; a.k_new = fz->k; a.v_new = fz->v; a.rope_table = fz->rope_table;
    a.rope_max_pos = fz->rope_max_pos; a.q_rot_out = fz->q_rot_out;
    a.k_arena_w = fz->k_arena; a.v_arena_w = fz->v_arena;
  }
  a.early_inputs = dependent ? 1 : 0;
  if ((e = status_ptr(&a.status)) != cudaSuccess) return cuda_fail(e, "status word");

  const long long rows = static_cast<long long>(num_blocks) * num_kv_heads * block_size;
  CUtensorMap kmap, vmap, qmap;
  if ((rc = arena_map(&kmap, k_arena, dtype, head_dim, rows, 16))) return rc;
  if ((rc = arena_map(&vmap, v_arena, dtype, head_dim, rows, 16))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // decode class: query_len x group <= decode_max_rows, i.e. query_len <= qd.
  // The query lengths sum to num_tokens and none exceeds max_query_len, so
  // when num_tokens > (num_seqs - 1) x max_query_len + qd no sequence can be
  // of the decode class and the decode launch is left out.
  const long long qd = a.decode_max_rows / a.group;
  const bool any_decode =
      qd >= 1 && static_cast<long long>(num_tokens) <= static_cast<long long>(num_seqs - 1) * max_query_len + qd;
  // prefill class: any sequence with more rows than the decode kernel takes
  const bool any_prefill = static_cast<long long>(max_query_len) * a.group > a.decode_max_rows;
  CUtensorMap kmap_p, vmap_p;
  if (any_prefill) {
    if ((rc = arena_map(&kmap_p, k_arena, dtype, head_dim, rows, block_size))) return rc;
    if ((rc = arena_map(&vmap_p, v_arena, dtype, head_dim, rows, block_size))) return rc;
    if ((rc = query_map(&qmap, fz ? fz->q : q_rot, dtype, head_dim, num_q_heads, num_tokens, a.group))) return rc;
  }
  SideStream* side = any_decode && any_prefill ? side_stream() : nullptr;
  if (side) {  // the prefill kernel beside the decode kernel
    a.beside_decode = 1;
    if ((e = cudaEventRecord(side->fork, s)) != cudaSuccess) return cuda_fail(e, "side stream fork");
    if ((e = cudaStreamWaitEvent(side->stream, side->fork, 0)) != cudaSuccess) return cuda_fail(e, "side stream fork");
    if ((e = launch_prefill(a, kmap_p, vmap_p, qmap, side->stream)) != cudaSuccess)
      return cuda_fail(e, "prefill kernel launch");
    if ((e = cudaEventRecord(side->join, side->stream)) != cudaSuccess) return cuda_fail(e, "side stream join");
  }
  if (any_decode) {
    if (a.ws_counters && (e = cudaMemsetAsync(a.ws_counters, 0, plan.counter_bytes, s)) != cudaSuccess)
      return cuda_fail(e, "clearing split counters");
    if ((e = launch_decode(a, kmap, vmap, s)) != cudaSuccess) return cuda_fail(e, "decode kernel launch");
  }
  if (side) {
    if ((e = cudaStreamWaitEvent(s, side->join, 0)) != cudaSuccess) return cuda_fail(e, "side stream join");
  } else if (any_prefill) {
    if ((e = launch_prefill(a, kmap_p, vmap_p, qmap, s)) != cudaSuccess) return cuda_fail(e, "prefill kernel launch");
  }
  return KSHIPRA_OK;
}


}  // namespace

// The same helpers for the other translation units (internal.h).
namespace kshipra {
void api_clear_error() { g_last_error[0] = 0; }
int api_fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}
int api_cuda_fail(cudaError_t e, const char* what) { return cuda_fail(e, what); }
cudaError_t api_status_ptr(unsigned** out) { return status_ptr(out); }
bool api_side_streams(bool on) {
  const bool was = !g_side_off;
  g_side_off = !on;
  return was;
}
}  // namespace kshipra

// ===========================================================================
extern "C" {

size_t kshipra_kv_bytes_per_token(int num_layers, int num_kv_heads, int head_dim, int dtype) {
  if (num_layers <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  if (dtype != KSHIPRA_DTYPE_F16 && dtype != KSHIPRA_DTYPE_BF16) return 0;
  const size_t elem = 2;  // both storage types are 16-bit
  return 2 * static_cast<size_t>(num_layers) * num_kv_heads * head_dim * elem;
}

int kshipra_rope_table_build(float* host_out, int max_pos, int head_dim, double theta) {
  if (!host_out) return fail(KSHIPRA_ERR_INVALID_ARG, "host_out is NULL");
  if (max_pos < 0 || head_dim < 2 || (head_dim & 1) || !(theta > 0.0))
    return fail(KSHIPRA_ERR_INVALID_ARG, "bad rope table shape (max_pos %d, head_dim %d, theta %g)", max_pos,
                head_dim, theta);
  const int half = head_dim / 2;
  for (int i = 0; i < half; ++i) {
    const double inv_freq = std::pow(theta, -2.0 * i / head_dim);
    for (long p = 0; p < max_pos; ++p) {
      const double angle = static_cast<double>(p) * inv_freq;
      host_out[(p * half + i) * 2] = static_cast<float>(std::cos(angle));
      host_out[(p * half + i) * 2 + 1] = static_cast<float>(std::sin(angle));
    }
  }
  return KSHIPRA_OK;
}

int kshipra_set_option(int option, int value) {
  switch (option) {
    case KSHIPRA_OPT_SPLIT_TOKENS:
      if (value < 0 || value % 64)
        return fail(KSHIPRA_ERR_INVALID_ARG, "split tokens %d must be 0 or a positive multiple of 64", value);
      g_opt_split_tokens = value;
      return KSHIPRA_OK;
    case KSHIPRA_OPT_DECODE_MAX_ROWS:
      if (value < 0 || value > kDecodeMaxRows)
        return fail(KSHIPRA_ERR_INVALID_ARG, "decode max rows %d not in [0, %d]", value, kDecodeMaxRows);
      g_opt_decode_max_rows = value;
      return KSHIPRA_OK;
    default:
      return fail(KSHIPRA_ERR_INVALID_ARG, "unknown option %d", option);
  }
}

const char* kshipra_status_string(int code) {
  switch (code) {
    case KSHIPRA_OK: return "ok";
    case KSHIPRA_ERR_INVALID_ARG: return "invalid argument";
    case KSHIPRA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case KSHIPRA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case KSHIPRA_ERR_CUDA: return "CUDA error";
    case KSHIPRA_ERR_OUT_OF_BLOCKS: return "not enough free blocks";
    default: return "unknown status";
  }
}

const char* kshipra_last_error(void) { return g_last_error; }

int kshipra_device_status(int32_t* code_out, void* stream) {
  if (!code_out) return fail(KSHIPRA_ERR_INVALID_ARG, "code_out is NULL");
  unsigned* st = nullptr;
  cudaError_t e = status_ptr(&st);
  if (e != cudaSuccess) return cuda_fail(e, "status word");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  if ((e = cudaMemcpyAsync(&v, st, sizeof v, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
      (e = cudaMemsetAsync(st, 0, sizeof v, s)) != cudaSuccess || (e = cudaStreamSynchronize(s)) != cudaSuccess)
    return cuda_fail(e, "reading the status word");
  *code_out = static_cast<int32_t>(v);
  return KSHIPRA_OK;
}

int kshipra_kv_append_rope(const void* q, const void* k, const void* v, void* q_rot, void* k_arena,
                           void* v_arena, const int32_t* block_tables, const int32_t* query_start_loc,
                           const int32_t* positions, const float* rope_table, int rope_max_pos, int num_seqs,
                           int num_tokens, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int max_blocks_per_seq, int num_blocks, int dtype, void* stream) {
  g_last_error[0] = 0;
  AppendArgs a{};
  int rc = append_prepare(&a, q, k, v, q_rot, k_arena, v_arena, block_tables, query_start_loc, positions, rope_table,
                          rope_max_pos, num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
                          max_blocks_per_seq, num_blocks, dtype);
  if (rc || num_tokens == 0) return rc;
  const cudaError_t e = launch_append_rope(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append kernel launch");
  return KSHIPRA_OK;
}

int kshipra_paged_attention_workspace_size(int num_seqs, int num_tokens, int max_context_len, int num_q_heads,
                                           int num_kv_heads, int head_dim, int sm_count, size_t* bytes_out) {
  g_last_error[0] = 0;
  if (!bytes_out) return fail(KSHIPRA_ERR_INVALID_ARG, "bytes_out is NULL");
  if (num_seqs < 0 || num_tokens < 0 || max_context_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || sm_count < 0)
    return fail(KSHIPRA_ERR_INVALID_ARG, "bad workspace query arguments");
  if (sm_count == 0) {
    cudaError_t e = sm_count_current(&sm_count);
    if (e != cudaSuccess) return cuda_fail(e, "SM count");
  }
  *bytes_out = plan_workspace(num_seqs, num_tokens, max_context_len, num_q_heads, num_kv_heads, head_dim, sm_count)
                   .total;
  return KSHIPRA_OK;
}

int kshipra_paged_attention(void* out, const void* q_rot, const void* k_arena, const void* v_arena,
                            const int32_t* block_tables, const int32_t* context_lens,
                            const int32_t* query_start_loc, const int32_t* positions, int num_seqs,
                            int num_tokens, int max_query_len, int max_context_len, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                            int num_blocks, float scale, int dtype, void* workspace, size_t workspace_bytes,
                            void* stream) {
  g_last_error[0] = 0;
  return attention_impl(out, q_rot, k_arena, v_arena, block_tables, context_lens, query_start_loc, positions,
                        num_seqs, num_tokens, max_query_len, max_context_len, num_q_heads, num_kv_heads, head_dim,
                        block_size, max_blocks_per_seq, num_blocks, scale, dtype, workspace, workspace_bytes, stream,
                        nullptr);
}

int kshipra_decode_step(void* out, const void* q, const void* k, const void* v, void* q_rot, void* k_arena,
                       void* v_arena, const int32_t* block_tables, const int32_t* context_lens,
                       const int32_t* query_start_loc, const int32_t* positions, const float* rope_table,
                       int rope_max_pos, int num_seqs, int num_tokens, int max_query_len, int max_context_len,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                       int num_blocks, float scale, int dtype, void* workspace, size_t workspace_bytes,
                       void* stream) {
  g_last_error[0] = 0;
  int rc = check_heads(num_q_heads, num_kv_heads, head_dim, block_size, dtype);
  if (rc) return rc;
  if (rope_max_pos <= 0) return fail(KSHIPRA_ERR_INVALID_ARG, "rope_max_pos must be positive");
  if (num_tokens > 0 && (!q || !k || !v || !rope_table))
    return fail(KSHIPRA_ERR_INVALID_ARG, "a required pointer is NULL");
  const void* vec[] = {q, k, v, q_rot, rope_table};
  for (const void* p : vec)
    if (p && !aligned(p, 16)) return fail(KSHIPRA_ERR_INVALID_ARG, "data pointers must be 16-byte aligned");
  if (q_rot && (q_rot == out || q_rot == q)) return fail(KSHIPRA_ERR_INVALID_ARG, "q_rot must not alias out or q");
  const int group = num_q_heads / num_kv_heads;
  if (static_cast<long long>(max_query_len) * group > g_opt_decode_max_rows) {
    // rows for the tensor-core prefill kernels: the K/V append, then attention
    // kernels that rotate q themselves (q_rot optional); with head_dim 128
    // they start while the append finishes (launched as its programmatic
    // dependents).  Every host check runs before the append is enqueued.
    const bool dependent = head_dim == 128;
    const FusedInputs fz{q, nullptr, nullptr, rope_table, rope_max_pos, q_rot, k_arena, v_arena};
    if ((rc = attention_impl(out, q_rot, k_arena, v_arena, block_tables, context_lens, query_start_loc, positions,
                             num_seqs, num_tokens, max_query_len, max_context_len, num_q_heads, num_kv_heads,
                             head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype, workspace,
                             workspace_bytes, stream, &fz, dependent, true)))
      return rc;
    AppendArgs ap{};
    if ((rc = append_prepare(&ap, nullptr, k, v, nullptr, k_arena, v_arena, block_tables, query_start_loc, positions,
                             rope_table, rope_max_pos, num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim,
                             block_size, max_blocks_per_seq, num_blocks, dtype)))
      return rc;
    if (num_tokens > 0) {
      const cudaError_t e = launch_append_rope(ap, static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_fail(e, "append kernel launch");
    }
    return attention_impl(out, q_rot, k_arena, v_arena, block_tables, context_lens, query_start_loc, positions,
                          num_seqs, num_tokens, max_query_len, max_context_len, num_q_heads, num_kv_heads, head_dim,
                          block_size, max_blocks_per_seq, num_blocks, scale, dtype, workspace, workspace_bytes, stream,
                          &fz, dependent, false);
  }
  const FusedInputs fz{q, k, v, rope_table, rope_max_pos, q_rot, k_arena, v_arena};
  return attention_impl(out, q_rot, k_arena, v_arena, block_tables, context_lens, query_start_loc, positions,
                        num_seqs, num_tokens, max_query_len, max_context_len, num_q_heads, num_kv_heads, head_dim,
                        block_size, max_blocks_per_seq, num_blocks, scale, dtype, workspace, workspace_bytes, stream,
                        &fz);
}

}  // extern "C"
