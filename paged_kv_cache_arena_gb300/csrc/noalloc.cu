// kshipra_paged_attention_noalloc: paged attention for callers that cannot
// allocate device memory.
//
// Some callers can't call cudaMalloc or hand over a workspace: a server that
// reserved all free device memory up front for its KV arena (any later
// cudaMalloc would fail), a framework whose own allocator owns every device
// byte and forbids side allocations, or a latency-critical loop that must not
// pay cudaMalloc's implicit device-wide synchronisation.  This entry point
// runs the same computation as kshipra_paged_attention, but its split-KV
// partials live in a fixed scratch array that belongs to the library.
//
// The scratch array is a file-scope __device__ variable of
// KSHIPRA_NOALLOC_SCRATCH_BYTES bytes.  Every GPU on which the library is
// loaded holds it until the process exits.  In host code its name only stands
// in for the symbol; its device address is looked up once per device with
// cudaGetSymbolAddress (the first call on a device does this set-up, so make
// that first call before any stream capture) and passed to the kernels.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KSHIPRA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up on the
// first call made with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int kshipra_paged_attention_noalloc(void* out, const void* q_rot, const void* k_arena,
                                               const void* v_arena, const int32_t* block_tables,
                                               const int32_t* context_lens, const int32_t* query_start_loc,
                                               const int32_t* positions, int num_seqs, int num_tokens,
                                               int max_query_len, int max_context_len, int num_q_heads,
                                               int num_kv_heads, int head_dim, int block_size,
                                               int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                                               void* stream) {
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return kshipra::api_cuda_fail(e, "looking up the no-alloc scratch address");
  // The workspace check of kshipra_paged_attention rejects sizes whose split
  // partials exceed the scratch (KSHIPRA_ERR_WORKSPACE_TOO_SMALL, message in
  // kshipra_last_error) before anything is launched.  Every partial the
  // kernels read is written earlier in the same call, so nothing left by a
  // previous call needs clearing.  The call creates nothing either: a mixed
  // batch runs its kernels one after the other on the caller's stream
  // instead of on a side stream made on first use.
  const bool side_was_on = kshipra::api_side_streams(false);
  const int rc = kshipra_paged_attention(out, q_rot, k_arena, v_arena, block_tables, context_lens, query_start_loc,
                                         positions, num_seqs, num_tokens, max_query_len, max_context_len,
                                         num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                         num_blocks, scale, dtype, scratch, KSHIPRA_NOALLOC_SCRATCH_BYTES, stream);
  kshipra::api_side_streams(side_was_on);
  return rc;
}
