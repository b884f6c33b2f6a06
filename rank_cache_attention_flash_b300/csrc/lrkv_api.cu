// C-ABI host layer of liblrkv: argument validation, RoPE frequency table,
// TMA descriptors over the paged pools, split planning and dispatch to the
// bf16 (tensor-core) or fp32 kernels. Allocates nothing and keeps no state.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "lrkv.h"
#include "lrkv_testing.h"
#include "lrkv_device.cuh"
#include "lrkv_internal.h"

namespace lrkv {

void rope_freqs(const lrkv_config& cfg, RopeFreqs* f) {
  // the table of the last (base, d) seen by this host thread is reused
  thread_local float last_base = 0.f;
  thread_local int last_d = 0;
  thread_local RopeFreqs last;
  if (cfg.rope_base != last_base || cfg.head_dim != last_d) {
    std::memset(&last, 0, sizeof(last));
    const int half = cfg.head_dim / 2;
    for (int j = 0; j < half && j < 64; ++j) {
      const double th = std::pow(static_cast<double>(cfg.rope_base), -2.0 * j / cfg.head_dim);
      const float hi = static_cast<float>(th);
      last.hi[j] = hi;
      last.lo[j] = static_cast<float>(th - static_cast<double>(hi));
    }
    last_base = cfg.rope_base;
    last_d = cfg.head_dim;
  }
  *f = last;
}

namespace {
std::atomic<int> g_decode_test_stall{0};
}  // namespace

int decode_test_stall() { return g_decode_test_stall.load(std::memory_order_relaxed); }

int device_sm_count() {
  thread_local int last_dev = -1, last_n = 0;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev == last_dev) return last_n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  last_dev = dev;
  last_n = n;
  return n;
}

bool ensure_smem_attr(const void* func, int bytes) {
  // (kernel, device, bytes) triples already applied; a handful of kernels
  // times the devices in the process, so a linear scan is enough.
  struct Entry {
    const void* func;
    int dev;
    int bytes;
  };
  static std::mutex mu;
  static Entry done[256];
  static int n_done = 0;
  thread_local Entry last{nullptr, -1, 0};  // this host thread's last success: no lock
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (last.func == func && last.dev == dev && last.bytes >= bytes) return true;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i].func == func && done[i].dev == dev && done[i].bytes >= bytes) {
      last = done[i];
      return true;
    }
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return false;
  if (n_done < 256) done[n_done++] = Entry{func, dev, bytes};
  last = Entry{func, dev, bytes};
  return true;
}

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled raw_encoder() {
  static const EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiled>(p);
    return static_cast<EncodeTiled>(nullptr);
  }();
  return fn;
}

// A tensor-map encoding is a pure function of its arguments, and every call
// of an entry point encodes the same few maps again: each host thread keeps
// its last 16 encodings and copies a match instead of encoding.
CUresult encode_cached(CUtensorMap* map, CUtensorMapDataType dt, cuuint32_t rank, void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                       const cuuint32_t* es, CUtensorMapInterleave il, CUtensorMapSwizzle sw,
                       CUtensorMapL2promotion l2, CUtensorMapFloatOOBfill oob) {
  struct Key {
    int dt, il, sw, l2, oob;
    cuuint32_t rank;
    const void* base;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5], es[5];
  };
  struct Entry {
    Key key;
    CUtensorMap map;
    bool valid;
  };
  thread_local Entry cache[16];
  thread_local int next = 0;
  const EncodeTiled enc = raw_encoder();
  if (enc == nullptr) return CUDA_ERROR_NOT_INITIALIZED;
  if (rank < 1 || rank > 5) return enc(map, dt, rank, base, dims, strides, box, es, il, sw, l2, oob);
  Key k;
  std::memset(&k, 0, sizeof(k));
  k.dt = dt;
  k.il = il;
  k.sw = sw;
  k.l2 = l2;
  k.oob = oob;
  k.rank = rank;
  k.base = base;
  for (cuuint32_t i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    k.es[i] = es[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  for (const Entry& e : cache)
    if (e.valid && std::memcmp(&e.key, &k, sizeof(k)) == 0) {
      *map = e.map;
      return CUDA_SUCCESS;
    }
  const CUresult r = enc(map, dt, rank, base, dims, strides, box, es, il, sw, l2, oob);
  if (r == CUDA_SUCCESS) {
    cache[next].key = k;
    cache[next].map = *map;
    cache[next].valid = true;
    next = (next + 1) % 16;
  }
  return r;
}

EncodeTiled get_encoder() { return raw_encoder() != nullptr ? &encode_cached : nullptr; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

lrkv_status check_config(const lrkv_config* cfg) {
  if (cfg == nullptr) return LRKV_ERR_INVALID_ARG;
  if (cfg->hidden <= 0 || cfg->n_q_heads <= 0 || cfg->n_kv_heads <= 0 || cfg->head_dim <= 0 ||
      cfg->rank <= 0 || cfg->block_size <= 0 || !(cfg->rope_base > 0.f))
    return LRKV_ERR_INVALID_ARG;
  if (cfg->n_q_heads % cfg->n_kv_heads != 0) return LRKV_ERR_INVALID_ARG;
  if (cfg->dtype != LRKV_BF16 && cfg->dtype != LRKV_FP32) return LRKV_ERR_UNSUPPORTED;
  if (cfg->block_size != kBlock) return LRKV_ERR_UNSUPPORTED;
  if (cfg->head_dim != 64 && cfg->head_dim != 128) return LRKV_ERR_UNSUPPORTED;
  if (cfg->rank != 8 && cfg->rank != 16 && cfg->rank != 32 && cfg->rank != 64)
    return LRKV_ERR_UNSUPPORTED;
  if (cfg->n_q_heads / cfg->n_kv_heads > 16) return LRKV_ERR_UNSUPPORTED;
  if (cfg->hidden % 64 != 0) return LRKV_ERR_UNSUPPORTED;
  if (cfg->lr_groups < 1) return LRKV_ERR_INVALID_ARG;
  if (cfg->lr_groups > 64) return LRKV_ERR_UNSUPPORTED;
  if (cfg->kv_codec != LRKV_CODEC_NONE && cfg->kv_codec != LRKV_CODEC_POLYKV) return LRKV_ERR_INVALID_ARG;
  if (cfg->kv_codec == LRKV_CODEC_POLYKV && cfg->dtype != LRKV_BF16) return LRKV_ERR_UNSUPPORTED;
  return LRKV_OK;
}

// positions must stay below 2^20 (RoPE argument reduction range)
constexpr int64_t kMaxPositions = int64_t(1) << 20;

lrkv_status check_pool(const lrkv_config& cfg, const void* base_pool, const void* lr_pool,
                       int64_t num_blocks, int max_blocks) {
  if (base_pool == nullptr || lr_pool == nullptr) return LRKV_ERR_INVALID_ARG;
  if (!aligned16(base_pool) || !aligned16(lr_pool)) return LRKV_ERR_INVALID_ARG;
  if (num_blocks <= 0 || max_blocks <= 0) return LRKV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_blocks) * kBlock > kMaxPositions) return LRKV_ERR_UNSUPPORTED;
  // TMA row coordinates are int32
  if (num_blocks * 2 * cfg.n_kv_heads * kBlock > INT32_MAX) return LRKV_ERR_UNSUPPORTED;
  return LRKV_OK;
}

}  // namespace

// The 8-level Lloyd-Max quantiser for N(0, 1): Lloyd's iteration (thresholds
// at the midpoints of neighbouring centroids, centroids at the conditional
// means of their cells) in double precision, made exactly symmetric, rounded
// to float once. Computed on first use.
Codec make_polykv_codec() {
  constexpr int kL = 8;
  const double kInvSqrt2Pi = 0.39894228040143267794;
  auto pdf = [&](double x) { return std::isinf(x) ? 0.0 : kInvSqrt2Pi * std::exp(-0.5 * x * x); };
  auto upper = [](double x) { return 0.5 * std::erfc(x / std::sqrt(2.0)); };  // P(X > x)
  double c[kL], t[kL + 1];
  for (int k = 0; k < kL; ++k) c[k] = -2.0 + 4.0 * k / (kL - 1);
  for (int it = 0; it < 20000; ++it) {
    t[0] = -INFINITY;
    t[kL] = INFINITY;
    for (int k = 1; k < kL; ++k) t[k] = 0.5 * (c[k - 1] + c[k]);
    double diff = 0.0;
    for (int k = 0; k < kL; ++k) {
      const double mass = upper(t[k]) - upper(t[k + 1]);
      const double next = (pdf(t[k]) - pdf(t[k + 1])) / mass;
      diff = std::max(diff, std::fabs(next - c[k]));
      c[k] = next;
    }
    if (diff < 1e-15) break;
  }
  Codec q{};
  for (int k = 0; k < kL; ++k) q.centroid[k] = static_cast<float>(0.5 * (c[k] - c[kL - 1 - k]));
  for (int k = 0; k + 1 < kL; ++k) {
    const double a = 0.5 * (c[k] - c[kL - 1 - k]), b = 0.5 * (c[k + 1] - c[kL - 2 - k]);
    q.threshold[k] = static_cast<float>(0.5 * (a + b));
  }
  return q;
}

bool make_pool_maps(const lrkv_config& cfg, const void* base_pool, const void* lr_pool,
                    int64_t num_blocks, CUtensorMap* base_map, CUtensorMap* lr_map) {
  EncodeTiled enc = get_encoder();
  if (enc == nullptr) return false;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cfg.head_dim),
                                static_cast<cuuint64_t>(num_blocks) * 2 * cfg.n_kv_heads * kBlock};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cfg.head_dim) * 2};
    const cuuint32_t box[2] = {64, kBlock};
    const cuuint32_t es[2] = {1, 1};
    if (enc(base_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base_pool), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  if (lr_map == nullptr) return true;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(lr_width(cfg)),
                                static_cast<cuuint64_t>(num_blocks) * 2 * kBlock};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lr_width(cfg)) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(cfg.rank), kBlock};
    const cuuint32_t es[2] = {1, 1};
    CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (cfg.rank == 16) sw = CU_TENSOR_MAP_SWIZZLE_32B;
    if (cfg.rank == 32) sw = CU_TENSOR_MAP_SWIZZLE_64B;
    if (cfg.rank == 64) sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if (enc(lr_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(lr_pool), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

// 2-D map over a bf16 matrix whose rows hold `inner` elements `row_stride`
// bytes apart; box {box_inner, box_rows} with the swizzle matching a box row
// of `swizzle_span` bytes (128, 64, 32; anything else: none). Coordinates past
// the matrix read as zero.
bool make_bf16_2d_map(const void* base, int64_t inner, int64_t rows, int64_t row_stride, int box_inner,
                      int box_rows, int swizzle_span, CUtensorMap* map) {
  EncodeTiled enc = get_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle_span == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (swizzle_span == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  if (swizzle_span == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Low-rank pool map whose box is `box_cols` wide (>= rank): the columns past
// the rank read as zero (out-of-bounds fill), so a rank-8 tile lands in smem
// as a 16-column tile; rows of box_cols * 2 bytes with the matching swizzle.
bool make_lr_map(const lrkv_config& cfg, const void* lr_pool, int64_t num_blocks, int box_cols,
                 CUtensorMap* lr_map) {
  EncodeTiled enc = get_encoder();
  if (enc == nullptr || box_cols < cfg.rank) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(lr_width(cfg)),
                              static_cast<cuuint64_t>(num_blocks) * 2 * kBlock};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lr_width(cfg)) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), kBlock};
  const cuuint32_t es[2] = {1, 1};
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_32B;
  if (box_cols == 32) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  if (box_cols == 64) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  return enc(lr_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(lr_pool), dims, strides,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_bk_map(const lrkv_config& cfg, const void* B_K, int n_adapters, CUtensorMap* map) {
  EncodeTiled enc = get_encoder();
  if (enc == nullptr || n_adapters < 1) return false;
  const cuuint64_t d = static_cast<cuuint64_t>(cfg.head_dim);
  const cuuint64_t dims[3] = {d, static_cast<cuuint64_t>(cfg.n_kv_heads),
                              static_cast<cuuint64_t>(n_adapters) * cfg.rank};
  const cuuint64_t strides[2] = {d * 2, d * 2 * cfg.n_kv_heads};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(cfg.rank)};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(B_K), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D maps that load a run of `nb` consecutive blocks of one (K|V, kv head)
// chunk, or of one low-rank plane, in a single copy. Base pool dims: (d,
// 16 rows, 2 * Hkv chunks of a block, blocks), box {64, 16, 1, nb}; low-rank
// pool dims: (r, 16 rows, 2 planes, blocks), box {lr_cols, 16, 1, nb}. The
// copy lands as nb * 16 consecutive rows in shared memory, swizzled like the
// per-block maps.
bool make_run_maps(const lrkv_config& cfg, const void* base_pool, const void* lr_pool,
                   int64_t num_blocks, int nb, int lr_cols, CUtensorMap* base_map,
                   CUtensorMap* lr_map) {
  EncodeTiled enc = get_encoder();
  if (enc == nullptr || lr_cols < cfg.rank) return false;
  const cuuint64_t d = static_cast<cuuint64_t>(cfg.head_dim);
  {
    const cuuint64_t dims[4] = {d, kBlock, static_cast<cuuint64_t>(2 * cfg.n_kv_heads),
                                static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[3] = {d * 2, d * 2 * kBlock, d * 2 * kBlock * 2 * cfg.n_kv_heads};
    const cuuint32_t box[4] = {64, kBlock, 1, static_cast<cuuint32_t>(nb)};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(base_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base_pool), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  {
    const cuuint64_t r = static_cast<cuuint64_t>(lr_width(cfg));
    const cuuint64_t dims[4] = {r, kBlock, 2, static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[3] = {r * 2, r * 2 * kBlock, r * 2 * kBlock * 2};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(lr_cols), kBlock, 1, static_cast<cuuint32_t>(nb)};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_32B;
    if (lr_cols == 32) sw = CU_TENSOR_MAP_SWIZZLE_64B;
    if (lr_cols == 64) sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if (enc(lr_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(lr_pool), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

}  // namespace lrkv

using namespace lrkv;

extern "C" {

const char* lrkv_status_string(lrkv_status s) {
  switch (s) {
    case LRKV_OK: return "LRKV_OK";
    case LRKV_ERR_INVALID_ARG: return "LRKV_ERR_INVALID_ARG";
    case LRKV_ERR_UNSUPPORTED: return "LRKV_ERR_UNSUPPORTED";
    case LRKV_ERR_CUDA: return "LRKV_ERR_CUDA";
    case LRKV_ERR_INDEX: return "LRKV_ERR_INDEX";
    case LRKV_ERR_TIMEOUT: return "LRKV_ERR_TIMEOUT";
    case LRKV_ERR_WORKSPACE: return "LRKV_ERR_WORKSPACE";
  }
  return "LRKV_UNKNOWN_STATUS";
}

int32_t lrkv_version(void) { return 20200; }

size_t lrkv_base_pool_block_bytes(const lrkv_config* cfg) {
  if (check_config(cfg) != LRKV_OK) return 0;
  return base_block_bytes(*cfg);
}

void lrkv_testing_set_decode_stall(int32_t enable) {
  g_decode_test_stall.store(enable != 0 ? 1 : 0, std::memory_order_relaxed);
}

namespace {

lrkv_status append_common(const lrkv_config* cfg, const void* X_base, const void* X_lr, int32_t T,
                          const int32_t* positions, const int32_t* seq_rows, const int32_t* block_tables,
                          int32_t num_seqs, int32_t max_blocks, const void* W_cat, void* base_pool,
                          void* lr_pool, int64_t num_blocks, int32_t* dev_status, lrkv_stream_t stream) {
  lrkv_status st = check_config(cfg);
  if (st != LRKV_OK) return st;
  if (T < 0 || num_seqs < 0) return LRKV_ERR_INVALID_ARG;
  if (T == 0) return LRKV_OK;
  if ((X_base == nullptr && X_lr == nullptr) || positions == nullptr || seq_rows == nullptr ||
      block_tables == nullptr || W_cat == nullptr || num_seqs == 0)
    return LRKV_ERR_INVALID_ARG;
  if ((X_base != nullptr && !aligned16(X_base)) || (X_lr != nullptr && !aligned16(X_lr)) || !aligned16(W_cat) ||
      !aligned4(positions) || !aligned4(seq_rows) || !aligned4(block_tables))
    return LRKV_ERR_INVALID_ARG;
  if ((st = check_pool(*cfg, base_pool, lr_pool, num_blocks, max_blocks)) != LRKV_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cfg->dtype == LRKV_FP32)
    return launch_append_fp32(*cfg, X_base, X_lr, T, positions, seq_rows, block_tables, num_seqs, max_blocks,
                              W_cat, base_pool, lr_pool, num_blocks, dev_status, s);
  return launch_append_bf16(*cfg, X_base, X_lr, T, positions, seq_rows, block_tables, num_seqs, max_blocks,
                            W_cat, base_pool, lr_pool, num_blocks, dev_status, s);
}

}  // namespace

lrkv_status lrkv_append(const lrkv_config* cfg, const void* X, int32_t T,
                        const int32_t* positions, const int32_t* seq_rows,
                        const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks,
                        const void* W_cat, void* base_pool, void* lr_pool, int64_t num_blocks,
                        int32_t* dev_status, lrkv_stream_t stream) {
  return append_common(cfg, X, X, T, positions, seq_rows, block_tables, num_seqs, max_blocks, W_cat,
                       base_pool, lr_pool, num_blocks, dev_status, stream);
}

lrkv_status lrkv_append_rebase(const lrkv_config* cfg, const void* X_base, const void* X_lr, int32_t T,
                               const int32_t* positions, const int32_t* seq_rows,
                               const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks,
                               const void* W_cat, void* base_pool, void* lr_pool, int64_t num_blocks,
                               int32_t* dev_status, lrkv_stream_t stream) {
  return append_common(cfg, X_base, X_lr, T, positions, seq_rows, block_tables, num_seqs, max_blocks, W_cat,
                       base_pool, lr_pool, num_blocks, dev_status, stream);
}

size_t lrkv_decode_workspace_bytes(const lrkv_config* cfg, int32_t num_queries, int32_t num_ctx,
                                   int32_t max_ctx_len, int32_t max_q_per_ctx) {
  if (check_config(cfg) != LRKV_OK || num_queries < 0 || num_ctx < 0 || max_ctx_len < 0 ||
      max_q_per_ctx < 0)
    return 0;
  if (cfg->dtype == LRKV_FP32 || num_queries == 0 || num_ctx == 0) return 0;
  DecodePlan plan;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  if (!plan_decode_bf16(*cfg, num_queries, num_ctx, max_ctx_len, max_q_per_ctx, sms, &plan))
    return 0;
  return plan.ws_bytes;
}

}  // extern "C"

namespace {

// A validated decode call, ready to launch (empty: nothing to do).
struct DecodeCall {
  bool empty = true;
  bool fp32 = false;
  DecodeArgs a{};
  DecodePlan plan{};
  int max_q_per_ctx = 0;
  void* workspace = nullptr;
};

lrkv_status prepare_decode(const lrkv_config* cfg, const void* q, int32_t num_queries,
                           const int32_t* ctx_q_start, int32_t num_ctx, const int32_t* adapter_ids,
                           const int32_t* block_tables, int32_t max_blocks, const int32_t* ctx_lens,
                           int32_t max_ctx_len, int32_t max_q_per_ctx, const void* base_pool,
                           const void* lr_pool, int64_t num_blocks, const void* B_K, const void* B_V,
                           int32_t n_adapters, float scale, void* out, void* workspace,
                           size_t workspace_bytes, int32_t* dev_status, DecodeCall* c) {
  lrkv_status st = check_config(cfg);
  if (st != LRKV_OK) return st;
  if (num_queries < 0 || num_ctx < 0 || n_adapters < 0 || max_ctx_len < 0 || max_q_per_ctx < 0)
    return LRKV_ERR_INVALID_ARG;
  if (num_queries == 0 || num_ctx == 0) return LRKV_OK;
  if (q == nullptr || ctx_q_start == nullptr || adapter_ids == nullptr || block_tables == nullptr ||
      ctx_lens == nullptr || out == nullptr)
    return LRKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned4(ctx_q_start) || !aligned4(adapter_ids) ||
      !aligned4(block_tables) || !aligned4(ctx_lens))
    return LRKV_ERR_INVALID_ARG;
  if ((B_K != nullptr && !aligned16(B_K)) || (B_V != nullptr && !aligned16(B_V)))
    return LRKV_ERR_INVALID_ARG;
  if ((B_K != nullptr || B_V != nullptr) && n_adapters == 0) return LRKV_ERR_INVALID_ARG;
  if (cfg->lr_groups > 1 && n_adapters > cfg->lr_groups) return LRKV_ERR_INVALID_ARG;
  if (max_ctx_len < 1 || max_q_per_ctx < 1 || !(scale == scale)) return LRKV_ERR_INVALID_ARG;
  if ((st = check_pool(*cfg, base_pool, lr_pool, num_blocks, max_blocks)) != LRKV_OK) return st;
  if (static_cast<int64_t>(max_ctx_len) > static_cast<int64_t>(max_blocks) * kBlock)
    return LRKV_ERR_INVALID_ARG;
  c->a = DecodeArgs{q, num_queries, ctx_q_start, num_ctx, adapter_ids, block_tables, max_blocks,
                    ctx_lens, max_ctx_len, base_pool, lr_pool, num_blocks, B_K, B_V, n_adapters,
                    scale, out, dev_status};
  c->max_q_per_ctx = max_q_per_ctx;
  c->fp32 = cfg->dtype == LRKV_FP32;
  if (!c->fp32) {
    const int sms = device_sm_count();
    if (sms <= 0) return LRKV_ERR_CUDA;
    if (!plan_decode_bf16(*cfg, num_queries, num_ctx, max_ctx_len, max_q_per_ctx, sms, &c->plan))
      return LRKV_ERR_UNSUPPORTED;
    if (workspace == nullptr || workspace_bytes < c->plan.ws_bytes || !aligned16(workspace))
      return LRKV_ERR_WORKSPACE;
    c->workspace = workspace;
  }
  c->empty = false;
  return LRKV_OK;
}

lrkv_status launch_decode_call(const lrkv_config& cfg, const DecodeCall& c, cudaStream_t s) {
  if (c.empty) return LRKV_OK;
  if (c.fp32) return launch_decode_fp32(cfg, c.a, c.max_q_per_ctx, s);
  return launch_decode_bf16(cfg, c.a, c.plan, c.workspace, s);
}

// A validated prefill call, ready to launch (empty: nothing to do).
struct PrefillCall {
  bool empty = true;
  bool fp32 = false;
  PrefillArgs a{};
};

lrkv_status prepare_prefill(const lrkv_config* cfg, const void* q, const int32_t* q_start,
                            int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                            const int32_t* seq_lens, int32_t max_seq_len, const int32_t* adapter_ids,
                            const int32_t* block_tables, int32_t max_blocks, const void* base_pool,
                            const void* lr_pool, int64_t num_blocks, const void* B_K, const void* B_V,
                            int32_t n_adapters, float scale, void* out, int32_t* dev_status,
                            PrefillCall* c) {
  lrkv_status st = check_config(cfg);
  if (st != LRKV_OK) return st;
  if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || max_seq_len < 0 || n_adapters < 0)
    return LRKV_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_q == 0) return LRKV_OK;
  if (q == nullptr || q_start == nullptr || seq_lens == nullptr || adapter_ids == nullptr ||
      block_tables == nullptr || out == nullptr)
    return LRKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned4(q_start) || !aligned4(seq_lens) ||
      !aligned4(adapter_ids) || !aligned4(block_tables))
    return LRKV_ERR_INVALID_ARG;
  if ((B_K != nullptr && !aligned16(B_K)) || (B_V != nullptr && !aligned16(B_V)))
    return LRKV_ERR_INVALID_ARG;
  if ((B_K != nullptr || B_V != nullptr) && n_adapters == 0) return LRKV_ERR_INVALID_ARG;
  if (cfg->lr_groups > 1 && n_adapters > cfg->lr_groups) return LRKV_ERR_INVALID_ARG;
  if (max_q_len < 1 || max_seq_len < max_q_len || !(scale == scale)) return LRKV_ERR_INVALID_ARG;
  if ((st = check_pool(*cfg, base_pool, lr_pool, num_blocks, max_blocks)) != LRKV_OK) return st;
  if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks) * kBlock)
    return LRKV_ERR_INVALID_ARG;
  c->a = PrefillArgs{q, q_start, num_seqs, total_q, max_q_len, seq_lens, max_seq_len, adapter_ids,
                     block_tables, max_blocks, base_pool, lr_pool, num_blocks, B_K, B_V, n_adapters,
                     scale, out, dev_status};
  c->fp32 = cfg->dtype == LRKV_FP32;
  c->empty = false;
  return LRKV_OK;
}

lrkv_status launch_prefill_call(const lrkv_config& cfg, const PrefillCall& c, cudaStream_t s) {
  if (c.empty) return LRKV_OK;
  if (c.fp32) return launch_prefill_fp32(cfg, c.a, s);
  return launch_prefill_bf16(cfg, c.a, s);
}

// The second stream of a mixed call and its two events, one set per device
// and host thread, created on first use and kept (a stream and two events of
// each device this thread calls on).
struct ForkJoin {
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool ok = false;
};

ForkJoin* fork_join() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  thread_local ForkJoin fj[64];
  ForkJoin& f = fj[dev];
  if (!f.ok) {
    if (f.side == nullptr && cudaStreamCreateWithFlags(&f.side, cudaStreamNonBlocking) != cudaSuccess) {
      f.side = nullptr;
      return nullptr;
    }
    if (f.fork == nullptr && cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming) != cudaSuccess) {
      f.fork = nullptr;
      return nullptr;
    }
    if (f.join == nullptr && cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming) != cudaSuccess) {
      f.join = nullptr;
      return nullptr;
    }
    f.ok = true;
  }
  return &f;
}

}  // namespace

extern "C" {

lrkv_status lrkv_attn_decode(const lrkv_config* cfg, const void* q, int32_t num_queries,
                             const int32_t* ctx_q_start, int32_t num_ctx,
                             const int32_t* adapter_ids, const int32_t* block_tables,
                             int32_t max_blocks, const int32_t* ctx_lens, int32_t max_ctx_len,
                             int32_t max_q_per_ctx, const void* base_pool, const void* lr_pool,
                             int64_t num_blocks, const void* B_K, const void* B_V,
                             int32_t n_adapters, float scale, void* out, void* workspace,
                             size_t workspace_bytes, int32_t* dev_status, lrkv_stream_t stream) {
  DecodeCall c;
  const lrkv_status st = prepare_decode(cfg, q, num_queries, ctx_q_start, num_ctx, adapter_ids, block_tables,
                                        max_blocks, ctx_lens, max_ctx_len, max_q_per_ctx, base_pool, lr_pool,
                                        num_blocks, B_K, B_V, n_adapters, scale, out, workspace,
                                        workspace_bytes, dev_status, &c);
  if (st != LRKV_OK) return st;
  return launch_decode_call(*cfg, c, reinterpret_cast<cudaStream_t>(stream));
}

size_t lrkv_prefill_workspace_bytes(const lrkv_config* cfg, int32_t num_seqs, int32_t total_q,
                                    int32_t max_q_len, int32_t max_seq_len) {
  (void)cfg;
  (void)num_seqs;
  (void)total_q;
  (void)max_q_len;
  (void)max_seq_len;
  return 0;
}

lrkv_status lrkv_attn_prefill(const lrkv_config* cfg, const void* q, const int32_t* q_start,
                              int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                              const int32_t* seq_lens, int32_t max_seq_len,
                              const int32_t* adapter_ids, const int32_t* block_tables,
                              int32_t max_blocks, const void* base_pool, const void* lr_pool,
                              int64_t num_blocks, const void* B_K, const void* B_V,
                              int32_t n_adapters, float scale, void* out, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, lrkv_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  PrefillCall c;
  const lrkv_status st = prepare_prefill(cfg, q, q_start, num_seqs, total_q, max_q_len, seq_lens, max_seq_len,
                                         adapter_ids, block_tables, max_blocks, base_pool, lr_pool, num_blocks,
                                         B_K, B_V, n_adapters, scale, out, dev_status, &c);
  if (st != LRKV_OK) return st;
  return launch_prefill_call(*cfg, c, reinterpret_cast<cudaStream_t>(stream));
}

lrkv_status lrkv_attn_mixed(const lrkv_config* cfg, const lrkv_decode_batch* dec,
                            const lrkv_prefill_batch* pre, const void* base_pool, const void* lr_pool,
                            int64_t num_blocks, const void* B_K, const void* B_V, int32_t n_adapters,
                            float scale, int32_t* dev_status, lrkv_stream_t stream) {
  DecodeCall dc;
  PrefillCall pc;
  lrkv_status st = check_config(cfg);
  if (st != LRKV_OK) return st;
  if (dec != nullptr &&
      (st = prepare_decode(cfg, dec->q, dec->num_queries, dec->ctx_q_start, dec->num_ctx, dec->adapter_ids,
                           dec->block_tables, dec->max_blocks, dec->ctx_lens, dec->max_ctx_len,
                           dec->max_q_per_ctx, base_pool, lr_pool, num_blocks, B_K, B_V, n_adapters, scale,
                           dec->out, dec->workspace, dec->workspace_bytes, dev_status, &dc)) != LRKV_OK)
    return st;
  if (pre != nullptr &&
      (st = prepare_prefill(cfg, pre->q, pre->q_start, pre->num_seqs, pre->total_q, pre->max_q_len,
                            pre->seq_lens, pre->max_seq_len, pre->adapter_ids, pre->block_tables,
                            pre->max_blocks, base_pool, lr_pool, num_blocks, B_K, B_V, n_adapters, scale,
                            pre->out, dev_status, &pc)) != LRKV_OK)
    return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dc.empty || pc.empty) {
    if ((st = launch_prefill_call(*cfg, pc, s)) != LRKV_OK) return st;
    return launch_decode_call(*cfg, dc, s);
  }
  // Both parts: the prefill on the caller's stream, the decode on a second
  // stream forked from it and joined back, so that the decode's CTAs fill the
  // SMs the prefill grid leaves idle (its last partial wave) instead of
  // waiting for the whole prefill.
  ForkJoin* fj = fork_join();
  if (fj == nullptr) return LRKV_ERR_CUDA;
  if (cudaEventRecord(fj->fork, s) != cudaSuccess || cudaStreamWaitEvent(fj->side, fj->fork, 0) != cudaSuccess)
    return LRKV_ERR_CUDA;
  const lrkv_status sp = launch_prefill_call(*cfg, pc, s);
  const lrkv_status sd = launch_decode_call(*cfg, dc, fj->side);
  // the join is recorded whatever the launches returned, so the caller's
  // stream never runs ahead of work still queued on the second stream
  if (cudaEventRecord(fj->join, fj->side) != cudaSuccess || cudaStreamWaitEvent(s, fj->join, 0) != cudaSuccess)
    return LRKV_ERR_CUDA;
  return sp != LRKV_OK ? sp : sd;
}

}  // extern "C"
