// Internal declarations shared by the C-ABI layer and the kernel translation
// units.  Not part of the public interface (include/pqkv.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pqkv.h"

namespace pqkv {

constexpr int kHeadDim = 128;
constexpr int kPageSize = 16;

struct AppendParams {
  const uint16_t* k;        // fp16 bits
  const uint16_t* v;
  int64_t k_stride;         // elements between tokens
  int64_t v_stride;
  const int64_t* slots;
  const float* k_scale;
  const float* v_scale;
  int32_t scale_per_head;
  int32_t num_tokens;
  int32_t num_kv_heads;
  uint8_t* pages;
  int64_t num_pages;
  uint16_t* row_scales;     // INT8_ROW: fp16 bits [num_pages][Hkv][8][4] after the codes
  int32_t* status;
};

struct AttnParams {
  const uint16_t* q;        // fp16 bits [B*q_len][Hq][128]
  uint16_t* out;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const float* k_scale;     // INT8_ROW: the fp16 row scales [num_pages][Hkv][8][4]
  const float* v_scale;
  int32_t* counters;        // [B*Hkv] merge tickets (workspace)
  float* part_o;            // [slots][RP][128] unnormalised partial outputs
  float* part_ml;           // [slots][2][RP]   running max (log2 units) and sum
  int32_t* status;
  int64_t num_pages;
  int32_t bt_stride;        // max_pages_per_seq
  int32_t num_seqs;
  int32_t q_len;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;            // num_q_heads / num_kv_heads
  int32_t rows;             // group * q_len
  int32_t scale_per_head;
  int32_t num_splits;       // 0: balanced shares, k >= 1: k partitions per (seq, head)
  float sm_scale_log2;      // log2(e) / sqrt(head_dim)
};

// Partial mode (one rank's share of a sequence's keys, for a decode context
// parallel split across GPUs): the keys of sequence s are its local cache;
// query i sits at local index q_pos[s] + i; the output is O / l in fp32 and
// the natural-log LSE m + ln l of every (query, q-head) row.
struct AttnPartialParams : AttnParams {
  const int32_t* q_pos;     // [B] local index of query 0's position
  float* out_o;             // [B*q_len][Hq][128]
  float* out_lse;           // [B*q_len][Hq]
};

// Sliding-window attention: query position p sees keys p - window + 1 .. p
// (window >= 1); the pages wholly before every query's window are never read.
struct AttnWindowParams : AttnParams {
  int32_t window;
};

// Test mode of the bounded waits: the feed of block `skip_block` does not
// issue the copy of that block's page `skip_page` (its position in the
// block's share), so the warp that owns the page waits for a tile that never
// comes; waits give up after 1 ms instead of 1 s.  Built only into the
// testing entry point.
struct AttnWaitTestParams : AttnParams {
  int32_t skip_block;
  int32_t skip_page;
};

// Host launchers (one per KV format), defined in the attention translation units.
cudaError_t launch_attention_fp16(const AttnParams& p, const CUtensorMap& map, int grid,
                                  int nt, bool pair, cudaStream_t stream);
cudaError_t launch_attention_e4m3(const AttnParams& p, const CUtensorMap& map, int grid,
                                  int nt, bool pair, cudaStream_t stream);
cudaError_t launch_attention_int8(const AttnParams& p, const CUtensorMap& map, int grid,
                                  int nt, bool pair, cudaStream_t stream);
cudaError_t launch_attention_int8_row(const AttnParams& p, const CUtensorMap& map, int grid,
                                      int nt, bool pair, cudaStream_t stream);
// Resident blocks per SM of the attention kernel for a KV format, n-tile
// count, block shape (pair: the 8-row decode as two 8-warp blocks per SM)
// and number of sequences (0 if the query fails).
int attention_blocks_per_sm_fp16(int nt, bool pair, int num_seqs);
int attention_blocks_per_sm_e4m3(int nt, bool pair, int num_seqs);
int attention_blocks_per_sm_int8(int nt, bool pair, int num_seqs);
int attention_blocks_per_sm_int8_row(int nt, bool pair, int num_seqs);

cudaError_t launch_attention_partial_fp16(const AttnPartialParams& p, const CUtensorMap& map,
                                          int grid, int nt, bool pair,
                                          cudaStream_t stream);
cudaError_t launch_attention_partial_e4m3(const AttnPartialParams& p, const CUtensorMap& map,
                                          int grid, int nt, bool pair,
                                          cudaStream_t stream);
cudaError_t launch_attention_partial_int8(const AttnPartialParams& p, const CUtensorMap& map,
                                          int grid, int nt, bool pair,
                                          cudaStream_t stream);
cudaError_t launch_attention_partial_int8_row(const AttnPartialParams& p, const CUtensorMap& map,
                                              int grid, int nt, bool pair,
                                          cudaStream_t stream);
cudaError_t launch_attention_window_fp16(const AttnWindowParams& p, const CUtensorMap& map,
                                         int grid, int nt, cudaStream_t stream);
cudaError_t launch_attention_window_e4m3(const AttnWindowParams& p, const CUtensorMap& map,
                                         int grid, int nt, cudaStream_t stream);
cudaError_t launch_attention_window_int8(const AttnWindowParams& p, const CUtensorMap& map,
                                         int grid, int nt, cudaStream_t stream);
cudaError_t launch_attention_window_int8_row(const AttnWindowParams& p, const CUtensorMap& map,
                                             int grid, int nt, cudaStream_t stream);
cudaError_t launch_attention_wait_test_e4m3(const AttnWaitTestParams& p, const CUtensorMap& map,
                                            int grid, int nt, cudaStream_t stream);
cudaError_t launch_lse_merge(const float* part_o, const float* part_lse, int num_parts,
                             int64_t rows, uint16_t* out, float* out_lse, cudaStream_t stream);

// Append launch shape: blocks of kAppendThreads threads, each thread takes
// kAppendUnroll 16-element vectors per pass with every load of the pass
// issued before the first encode (kAppendUnroll * 64 bytes in flight).
constexpr int kAppendThreads = 256;
constexpr int kAppendUnroll = 1;
cudaError_t launch_append(const AppendParams& p, int kv_dtype, int grid, cudaStream_t stream);
int append_blocks_per_sm(int kv_dtype);

// The arguments of one attention call (the shared part of the entry points).
struct AttnArgs {
  const void* q;
  const void* pages;
  int64_t num_pages;
  const int32_t* block_table;
  int32_t max_pages_per_seq;
  const int32_t* seq_lens;
  int32_t num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype;
  const float* k_scale;
  const float* v_scale;
  int32_t scale_per_head, num_splits, max_seq_len;
  int32_t window = 0;       // sliding window (0: none); only sizes the grid here
};

// Workspace carve-up of one call: merge counters, partial O, partial (m, l).
struct AttnPlan {
  int rows = 0, rp = 0, nt = 0;
  int64_t slots = 0;        // partial-result slots
  size_t counter_bytes = 0, o_bytes = 0, ml_bytes = 0, total = 0;
};

// Launch shape of one validated call: grid, row tiles, block shape (pair: the
// 8-row decode of a short context as two 8-warp blocks per SM) and the
// workspace it needs.
struct AttnLaunch {
  int grid = 0, nt = 0, rows = 0;
  bool pair = false;
  AttnPlan pl;
};

// Validate the arguments and size the launch (grid and workspace need) on the
// current device.  Queues nothing.  num_seqs == 0 returns PQKV_OK with an
// empty launch.
int plan_attention_launch(const AttnArgs& a, AttnLaunch* L);
// Check the workspace against the launch, encode the pool's TMA map and fill
// the kernel parameters (all but the outputs).  Queues nothing.
int bind_attention(const AttnArgs& a, const AttnLaunch& L, void* workspace,
                   size_t workspace_bytes, int32_t* status, AttnParams* p, CUtensorMap* map);
// Launch the attention kernel of the pool's format.
cudaError_t launch_attention(int kv_dtype, const AttnParams& p, const CUtensorMap& map, int grid,
                             int nt, bool pair, cudaStream_t stream);
// PQKV_EINVAL (after the size checks) when num_seqs > 0 and an output
// argument is missing or misaligned.
int check_output_args(const AttnArgs& a, bool bad_outputs);

inline int rows_padded(int rows) { return ((rows + 7) / 8) * 8; }

}  // namespace pqkv
