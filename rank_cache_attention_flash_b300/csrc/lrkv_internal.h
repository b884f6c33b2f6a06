// Internal interfaces between the C-ABI host layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "lrkv.h"

namespace lrkv {

struct RopeFreqs;  // lrkv_device.cuh

// Columns of one low-rank pool row: every group's r columns side by side.
inline int lr_width(const lrkv_config& cfg) { return cfg.lr_groups * cfg.rank; }

// Compressed base pool (LRKV_CODEC_POLYKV): per (block, kv head) one chunk of
//   Kq int8 [16][d] | Ks fp16 [16][d/32] | Vq u8 [16][3][d/8] | Vn fp32 [16]
__host__ __device__ constexpr int codec_chunk_bytes(int d) { return 23 * d + 64; }
__host__ __device__ constexpr int codec_k_bytes(int d) { return 17 * d; }      // Kq + Ks: what a K item copies per block
__host__ __device__ constexpr int codec_v_bytes(int d) { return 6 * d + 64; }  // Vq + Vn: what a V item copies per block
inline size_t base_block_bytes(const lrkv_config& cfg) {
  if (cfg.kv_codec == LRKV_CODEC_POLYKV) return static_cast<size_t>(cfg.n_kv_heads) * codec_chunk_bytes(cfg.head_dim);
  return static_cast<size_t>(2) * cfg.n_kv_heads * 16 * cfg.head_dim * (cfg.dtype == LRKV_FP32 ? 4 : 2);
}

// The 8-level Lloyd-Max quantiser for N(0,1) of the value codes, ascending.
struct Codec {
  float centroid[8];
  float threshold[7];
};
Codec make_polykv_codec();
inline const Codec& polykv_codec() {
  static const Codec c = make_polykv_codec();
  return c;
}

// Split plan of the bf16 decode kernel; a pure function of the sizes and the
// device's SM count, so the workspace query and the launch agree.
struct DecodePlan {
  int g;              // query heads per kv head
  int rows_per_item;  // query rows (query x head of the group) per work item
  int n_chunks;       // row chunks per (context, kv head)
  int n_splits;       // splits of each context's blocks
  int split_blocks;   // blocks per split
  int64_t n_items;    // num_ctx * n_chunks * n_splits * Hkv (one CTA each)
  int rebuild;        // 1: rebuild-mode kernel (one query per item, K_a rebuilt per tile)
  int smem_bytes;
  size_t ws_bytes;    // workspace: split partials
};

bool plan_decode_bf16(const lrkv_config& cfg, int num_queries, int num_ctx, int max_ctx_len,
                      int max_q_per_ctx, int sm_count, DecodePlan* plan);

struct DecodeArgs {
  const void* q;
  int num_queries;
  const int32_t* ctx_q_start;
  int num_ctx;
  const int32_t* adapter_ids;
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* ctx_lens;
  int max_ctx_len;
  const void* base_pool;
  const void* lr_pool;
  int64_t num_blocks;
  const void* B_K;
  const void* B_V;
  int n_adapters;
  float scale;
  void* out;
  int32_t* status;
};

// Host-built RoPE frequency table (theta_j split into two floats).
void rope_freqs(const lrkv_config& cfg, RopeFreqs* f);

// Tensor maps over the paged pools (lr_map may be NULL: base map only).
bool make_pool_maps(const lrkv_config& cfg, const void* base_pool, const void* lr_pool,
                    int64_t num_blocks, CUtensorMap* base_map, CUtensorMap* lr_map);
// 2-D map over a bf16 matrix [rows][inner] (rows row_stride bytes apart),
// box {box_inner, box_rows}, swizzle for box rows of swizzle_span bytes.
bool make_bf16_2d_map(const void* base, int64_t inner, int64_t rows, int64_t row_stride, int box_inner,
                      int box_rows, int swizzle_span, CUtensorMap* map);
// Low-rank pool map with a box of box_cols (>= rank) columns, zero-filled past the rank.
bool make_lr_map(const lrkv_config& cfg, const void* lr_pool, int64_t num_blocks, int box_cols,
                 CUtensorMap* lr_map);
// 3-D map over B_K [n_adapters][rank][Hkv][d] (bf16) with box {64, 1, rank}:
// one copy brings one adapter's rank rows of one kv head, 64 dims wide, as
// rank consecutive 128-byte rows with the 128-byte swizzle.
bool make_bk_map(const lrkv_config& cfg, const void* B_K, int n_adapters, CUtensorMap* map);
// 4-D maps copying a run of nb consecutive blocks per copy (base: one K|V
// chunk of one kv head; low-rank: one plane), box width lr_cols for the
// low-rank pool.
bool make_run_maps(const lrkv_config& cfg, const void* base_pool, const void* lr_pool,
                   int64_t num_blocks, int nb, int lr_cols, CUtensorMap* base_map,
                   CUtensorMap* lr_map);

lrkv_status launch_decode_bf16(const lrkv_config& cfg, const DecodeArgs& a,
                               const DecodePlan& plan, void* workspace, cudaStream_t stream);

// X_base feeds the base columns (K_base, V_base), X_lr the low-rank columns
// (L_K, L_V); a NULL source leaves that part of the pools untouched.
lrkv_status launch_append_bf16(const lrkv_config& cfg, const void* X_base, const void* X_lr, int T,
                               const int32_t* positions, const int32_t* seq_rows,
                               const int32_t* block_tables, int num_seqs, int max_blocks,
                               const void* W_cat, void* base_pool, void* lr_pool,
                               int64_t num_blocks, int32_t* status, cudaStream_t stream);

struct PrefillArgs {
  const void* q;
  const int32_t* q_start;
  int num_seqs;
  int total_q;
  int max_q_len;
  const int32_t* seq_lens;
  int max_seq_len;
  const int32_t* adapter_ids;
  const int32_t* block_tables;
  int max_blocks;
  const void* base_pool;
  const void* lr_pool;
  int64_t num_blocks;
  const void* B_K;
  const void* B_V;
  int n_adapters;
  float scale;
  void* out;
  int32_t* status;
};

lrkv_status launch_prefill_bf16(const lrkv_config& cfg, const PrefillArgs& a,
                                cudaStream_t stream);

// fp32 path (plain FMA, no tensor cores).
lrkv_status launch_append_fp32(const lrkv_config& cfg, const void* X_base, const void* X_lr, int T,
                               const int32_t* positions, const int32_t* seq_rows,
                               const int32_t* block_tables, int num_seqs, int max_blocks,
                               const void* W_cat, void* base_pool, void* lr_pool,
                               int64_t num_blocks, int32_t* status, cudaStream_t stream);
lrkv_status launch_decode_fp32(const lrkv_config& cfg, const DecodeArgs& a, int max_q_per_ctx,
                               cudaStream_t stream);
lrkv_status launch_prefill_fp32(const lrkv_config& cfg, const PrefillArgs& a,
                                cudaStream_t stream);

int device_sm_count();

// Test only (include/lrkv_testing.h): nonzero makes the next G-mode decode
// launches stall one bounded wait until it runs out.
int decode_test_stall();

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device. The attribute is per device, so it is set once per (kernel, device)
// pair, under a lock (concurrent first calls from several threads are safe).
bool ensure_smem_attr(const void* func, int bytes);

}  // namespace lrkv
