// Launch interface of the kernels behind pa.h (internal to libpa).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

// Element formats of the split kernel: FP16 Q with E4M3 or E5M2 K/V (head_dim
// 256, FP32 per-tensor scales), BF16 Q/K/V (head_dim 128 or 256), FP16 Q/K/V
// (head_dim 256).
enum KvFormat : int { kKvE4m3 = 0, kKvBf16 = 1, kKvE5m2 = 2, kKvF16 = 3, kKvBf16D256 = 4 };

// How the split kernel moves K and V rows into shared memory.
//   kKvLoadTma:    16-byte aligned bases and strides; TMA boxes with the
//                  128-byte swizzle, 256 row bytes per staged key.
//   kKvLoadWindow: bases 8 bytes past a 16-byte boundary, strides multiples of
//                  16; TMA boxes of 272-byte windows that start 8 bytes before
//                  each 256 row bytes (no swizzle).
//   kKvLoadCopy:   anything else 8-byte aligned; 8-byte cp.async by a warp.
enum KvLoad : int { kKvLoadCopy = 0, kKvLoadTma = 1, kKvLoadWindow = 2 };

// Split-KV kernel arguments (every element format).
struct SplitArgs {
  // 4-D views (row, KV head, slot, page) of K and V for the TMA loaders, with
  // boxes of 128, 64, 32 and 16 slots.  kKvLoadTma: byte elements, boxes of
  // 128 row bytes.  kKvLoadWindow: 16-bit elements from 8 bytes before the
  // base, boxes of 136 elements (272 bytes) of which the last 8 bytes lie
  // past the row's end (outside the view, so filled with zeros, not read).
  CUtensorMap k_maps[4];
  CUtensorMap v_maps[4];
  // kKvLoadTma only: 5-D byte views (row byte 0..127, KV head, slot, 128-byte
  // part of the key row, page) with one box of 128 slots x 2 parts: a whole
  // staging tile (128 keys x 256 row bytes) inside one page in one copy
  CUtensorMap k_map_tile;
  CUtensorMap v_map_tile;
  // 4-D element view of Q (d, query head, verify query, request) with boxes of
  // 64 elements x G heads x q_len queries (one 128-byte swizzled atom of the
  // packed tile); used when q_tma != 0
  CUtensorMap q_map;
  int q_tma;
  int kv_load;                 // KvLoad
  const void* q;               // FP16 or BF16 (the BF16 formats) [B][q_len][Hq][D]
  const uint8_t* k;            // K base: element (page, slot, head, d) at k + page*k_ps + slot*k_ts + head*k_hs
  const uint8_t* v;
  const int32_t* block_table;  // [B][mpr]
  const int32_t* ctx_lens;     // [B]
  const float* k_scale;        // 8-bit K/V formats only (E4M3, E5M2)
  const float* v_scale;        // 8-bit K/V formats only: the merged output is multiplied by *v_scale
  float2* panel_ml;            // (m in log2 units, l) per (item, row)
  float* panel_o;              // unnormalised O per (item, row, d); 8-bit paths: without v_scale
  void* out;                   // FP16, or BF16 for the BF16 formats: [B][q_len][Hq][D]
  float* lse;                  // nullable: natural-log LSE per output row
  uint32_t* status;
  uint32_t* bad;
  uint32_t* arrive;            // per request: softmax-group arrivals of its finished split items
  uint32_t* queue;             // next merge task
  uint32_t* done;              // CTAs that finished the call (the last one resets the per-call words)
  long long k_ps, k_ts, k_hs, v_ps, v_ts, v_hs;
  int B, Hkv, Hq, G, q_len, R, page_size, mpr, num_pages, max_ctx, s_max;
  long long wait_limit;  // pipeline wait bound in cycles (0: default)
  int withhold_q;        // test hook: never signal the Q tile, so the MMA wait runs out
};


// Causal prefill kernel arguments (FP16 Q/K/V, head_dim 256).  Work item
// it = ((s * B + b) * n_qt + qt) * Hq + h: query tile qt (128 queries) of
// query head h of request b against key split s (split_len keys).
struct PrefillArgs {
  // K: 4-D view (d, KV head, key, request), boxes of 64 d x 128 keys
  CUtensorMap k_map;
  // V: 5-D view (d within atom, key, atom, KV head, request), boxes of
  // 64 d x 32 keys x 4 atoms
  CUtensorMap v_map;
  const void* q;    // FP16 [B][q_len][Hq][256], contiguous
  float* part_o;    // FP32 partial O per (item tile, row, d), unnormalised
  float2* part_ml;  // (m in log2 units, l) per (item tile, row)
  uint32_t* status;
  int B, q_len, kv_len, Hq, Hkv, G, n_qt, split_len, num_splits, total_items;
  long long wait_limit;  // pipeline wait bound in cycles (0: default)
};

// Merge of the prefill split partials into FP16 output rows and the LSE.
struct PrefillMergeArgs {
  const float* part_o;
  const float2* part_ml;
  void* out;   // FP16 [B][q_len][Hq][256]
  float* lse;  // nullable, [B][q_len][Hq]
  int B, q_len, kv_len, Hq, n_qt, split_len, num_splits;
};

int prefill_smem_bytes();
cudaError_t launch_prefill(const PrefillArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_prefill_merge(const PrefillMergeArgs& m, cudaStream_t stream);

int split_smem_bytes();
cudaError_t launch_split(const SplitArgs& a, KvFormat fmt, int grid, cudaStream_t stream);
// per-format launchers behind launch_split (split_kv_<format>.cu)
cudaError_t launch_split_e4m3(const SplitArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_split_e5m2(const SplitArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_split_f16(const SplitArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_split_bf16_d128(const SplitArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_split_bf16_d256(const SplitArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_debug_worklist(const int32_t* ctx_lens, int B, int Hkv, int max_ctx, int32_t* items,
                                  int32_t max_items, int32_t* count, uint32_t* status, cudaStream_t stream);
cudaError_t launch_debug_gather(const uint8_t* base, long long ps, long long ts, long long hs, const int32_t* bt,
                                const int32_t* ctx_lens, int B, int Hkv, int page_size, int mpr, int num_pages,
                                int max_ctx, int row_bytes, uint8_t* dst, cudaStream_t stream);

}  // namespace pa
