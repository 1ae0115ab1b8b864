// Host-side interfaces between the C-ABI layer (api.cu) and the kernel
// translation units.  Every launcher enqueues on `stream` and returns the
// cudaError_t of the launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kshipra {

// Error reporting shared by the C-ABI entry points (api.cu): set the calling
// thread's last-error text and return the code; the device status word.
void api_clear_error();
int api_fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int api_cuda_fail(cudaError_t e, const char* what);
cudaError_t api_status_ptr(unsigned** out);
// Turns the calling thread's side streams (mixed batches run their prefill
// kernel beside the decode kernel) off or back on; returns the previous state.
bool api_side_streams(bool on);

// Rows of (token, q head) a decode unit handles at most: query_len x group.
constexpr int kDecodeMaxRows = 16;

struct AppendArgs {
  const void* q;
  const void* k;
  const void* v;
  void* q_rot;
  void* k_arena;
  void* v_arena;
  const int32_t* block_tables;
  const int32_t* query_start_loc;
  const int32_t* positions;
  const float* rope_table;
  int rope_max_pos;
  int num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks;
  int dtype;
  int sm_count;  // of the device the call runs on (sizes the grid)
  unsigned* status;
};

cudaError_t launch_append_rope(const AppendArgs& a, cudaStream_t stream);

// Shared by the decode, combine and prefill kernels.
struct AttnArgs {
  void* out;
  const void* q_rot;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start_loc;
  const int32_t* positions;
  float* ws_o;   // [max_splits][num_tokens][num_q_heads][head_dim] partial accumulators
  float* ws_ml;  // [max_splits][num_tokens][num_q_heads][2] partial (max, sum)
  unsigned* ws_counters;  // [num_seqs][num_kv_heads] finished splits, zeroed by the host each call
  uint64_t* ws_items;     // prefill (sequence, tile pair) entries, written by the planning kernel
  int* ws_item_count;     // work items = entries x num_kv_heads
  int max_items;          // capacity of ws_items (entries)
  int sm_count;           // CTAs of the persistent prefill kernel
  unsigned* status;
  int num_seqs, num_tokens, max_query_len, max_context_len;
  int num_q_heads, num_kv_heads, group, head_dim, block_size, max_blocks_per_seq, num_blocks;
  int split_tokens, max_splits;  // decode split size (keys) and count bound
  int decode_max_rows;           // query_len * group at or below this -> decode kernel
  int decode_ordered;            // decode CTAs take their units longest first (num_seqs <= kDecodeOrderedMaxSeqs)
  float scale_log2;              // scale * log2(e)
  int dtype;
  // fused step: when q_raw is set the attention kernels rotate the query rows
  // themselves (q_raw [T][Hq][d]; q_rot is then unused) and q_rot_out
  // (optional) receives the rotated q.  The decode kernel also writes the new
  // tokens' rotated K and raw V (k_new, v_new [T][Hkv][d]) into the arena
  // before reading it, unless k_new is NULL (a separate append wrote them).
  const void* q_raw;
  const void* k_new;
  const void* v_new;
  const float* rope_table;
  int rope_max_pos;
  void* q_rot_out;
  void* k_arena_w;
  void* v_arena_w;
  // every kernel of the library launches as a programmatic dependent of the
  // previous grid on the stream and waits for it before touching memory it
  // may write; with early_inputs set (the fused step, whose predecessor is
  // the library's own K/V append, which lets its dependents launch only after
  // its own predecessor has completed) the attention kernels read everything
  // but the arena before that wait
  int early_inputs;
  // mixed batch, head_dim 128: the pair kernel runs on a side stream beside
  // the decode kernel and keeps only the clusters its share of the call
  // needs (the rest leave at once, their SMs going to the decode kernel);
  // the decode kernel then launches as an ordinary dependent, so that it does
  // not take the SMs before the pair kernel has placed its clusters
  int beside_decode;
};

// Batches of at most this many sequences run their decode units longest
// first; each decode CTA finds its unit by scanning the batch's lengths, so
// the scan is kept to two rounds of 128 sequences.
constexpr int kDecodeOrderedMaxSeqs = 256;

// Split-KV decode (mma.sync on staged TMA tiles); the last split of each
// (sequence, kv head) to finish merges all partials.
cudaError_t launch_decode(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t stream);

// Upper bound on the prefill work-list entries of a call (pairs of 128-row
// query tiles per sequence).
int prefill_max_items(int num_seqs, int num_tokens, int num_q_heads, int num_kv_heads);

// Chunked prefill on tcgen05 / TMEM: planning kernel, then the persistent
// attention kernel.
cudaError_t launch_prefill(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const CUtensorMap& qmap, cudaStream_t stream);

// The same for head_dim 128 on CTA pairs (tcgen05 cta_group::2): planning
// kernel, then the persistent pair kernel.
cudaError_t launch_prefill_pair(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                const CUtensorMap& qmap, cudaStream_t stream);

}  // namespace kshipra
