// fp32 path: the same operations in plain fp32 FMA arithmetic (no tensor
// cores, no TF32), for workloads that keep every tensor in fp32.
//
// append: one CTA per token; each thread produces one K rotation pair, one V
//         column or one low-rank column from dot products over the hidden size.
// attention: one CTA per (query row, query head); keys are swept in chunks of
//         128 (one per thread): rebuild K_a[t] = K_base[t] + RoPE(L_K[t] B_K,a),
//         score, online softmax over the chunk, then O += P V_base and
//         O_lr += P L_V with threads over the output columns; at the end
//         out = (O + O_lr B_V,a) / l. Reordered exactly as the bf16 kernels
//         (LRAgent, arXiv 2602.01053, Abstract: Flash-LoRA-Attention).
#include <math_constants.h>

#include "lrkv_device.cuh"
#include "lrkv_internal.h"

namespace lrkv {
namespace {

constexpr int kChunk = 128;

struct Fp32AppendParams {
  const float* X_base;  // hidden states of the base columns (NULL: base part not written)
  const float* X_lr;    // hidden states of the low-rank columns (NULL: low-rank part not written)
  const float* W;       // [N][h]
  const int32_t* positions;
  const int32_t* seq_rows;
  const int32_t* block_tables;
  float* base_pool;
  float* lr_pool;
  int32_t* status;
  int64_t num_blocks;
  int h, Hkv, D, R, lrw, num_seqs, max_blocks;  // lrw: low-rank row width G * R
  RopeFreqs freqs;
};

__global__ void append_fp32_kernel(const __grid_constant__ Fp32AppendParams p) {
  extern __shared__ float xs[];
  const int t = blockIdx.x;
  const int s = __ldg(p.seq_rows + t), pos = __ldg(p.positions + t);
  if (s < 0 || s >= p.num_seqs || pos < 0 || pos >= p.max_blocks * kBlock) {
    if (threadIdx.x == 0) report(p.status, LRKV_ERR_INDEX);
    return;
  }
  const int blk = __ldg(p.block_tables + static_cast<int64_t>(s) * p.max_blocks + pos / kBlock);
  if (blk < 0 || blk >= p.num_blocks) {
    if (threadIdx.x == 0) report(p.status, LRKV_ERR_INDEX);
    return;
  }
  // xs[0, h): the base columns' hidden state; xs[h, 2h): the low-rank columns'
  for (int k = threadIdx.x; k < p.h; k += blockDim.x) {
    if (p.X_base != nullptr) xs[k] = p.X_base[static_cast<int64_t>(t) * p.h + k];
    if (p.X_lr != nullptr) xs[p.h + k] = p.X_lr[static_cast<int64_t>(t) * p.h + k];
  }
  __syncthreads();
  const int row = pos % kBlock, half = p.D / 2;
  const int kvc = p.Hkv * p.D;
  const int n_pairs = p.Hkv * half;
  const int units = n_pairs + kvc + 2 * p.lrw;
  auto dot = [&](int n) {
    const float* w = p.W + static_cast<int64_t>(n) * p.h;
    const float* x = n < 2 * kvc ? xs : xs + p.h;
    float acc = 0.f;
    for (int k = 0; k < p.h; ++k) acc = fmaf(w[k], x[k], acc);
    return acc;
  };
  for (int u = threadIdx.x; u < units; u += blockDim.x) {
    if ((u < n_pairs + kvc) ? p.X_base == nullptr : p.X_lr == nullptr) continue;
    if (u < n_pairs) {
      const int kv = u / half, j = u % half;
      const float x = dot(kv * p.D + j), y = dot(kv * p.D + j + half);
      const float2 cs = rope_cos_sin(pos, p.freqs.hi[j], p.freqs.lo[j]);
      float* dst = p.base_pool + (((static_cast<int64_t>(blk) * 2 + 0) * p.Hkv + kv) * kBlock + row) * p.D;
      dst[j] = x * cs.x - y * cs.y;
      dst[j + half] = y * cs.x + x * cs.y;
    } else if (u < n_pairs + kvc) {
      const int n = u - n_pairs;
      const int kv = n / p.D, j = n % p.D;
      p.base_pool[(((static_cast<int64_t>(blk) * 2 + 1) * p.Hkv + kv) * kBlock + row) * p.D + j] = dot(kvc + n);
    } else {
      const int n = u - n_pairs - kvc;  // [0, 2 G R)
      const int plane = n / p.lrw, k = n % p.lrw;
      p.lr_pool[((static_cast<int64_t>(blk) * 2 + plane) * kBlock + row) * p.lrw + k] = dot(2 * kvc + n);
    }
  }
}

struct Fp32AttnParams {
  const float* q;
  const int32_t* row_start;  // decode: ctx_q_start; prefill: q_start
  const int32_t* lens;       // keys per context / sequence
  const int32_t* adapter_ids;
  const int32_t* block_tables;
  const float* base_pool;
  const float* lr_pool;
  const float* B_K;
  const float* B_V;
  float* out;
  int32_t* status;
  int64_t num_blocks;
  int max_blocks, max_len, Hq, Hkv, D, R, n_adapters;
  int lrw, lr_groups;  // low-rank row width G * R; G > 1: adapter a reads group a
  int decode;  // 1: adapter per query row; 0: adapter per sequence
  float scale;
  RopeFreqs freqs;
};

// grid: (sequence / context, query row within it, query head)
__global__ void __launch_bounds__(kChunk) attn_fp32_kernel(const __grid_constant__ Fp32AttnParams p) {
  extern __shared__ float sm[];
  const int D = p.D, R = p.R;
  float* qv = sm;               // [D]
  float* sc = qv + D;           // [kChunk]
  float* acc = sc + kChunk;     // [D + R]
  float* red = acc + D + R;     // [kChunk / 32 + 2]
  const int c = blockIdx.x, qi = blockIdx.y, m = blockIdx.z;
  const int r0 = __ldg(p.row_start + c), r1 = __ldg(p.row_start + c + 1);
  if (r0 + qi >= r1) return;
  const int n = r0 + qi, nq = r1 - r0;
  const int len = __ldg(p.lens + c);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if ((!p.decode && len < nq) || len < 1 || len > p.max_len) {
    if (tid == 0) report(p.status, LRKV_ERR_INDEX);
    return;
  }
  int a = __ldg(p.adapter_ids + (p.decode ? n : c));
  if (a < -1 || a >= p.n_adapters) {
    if (tid == 0 && m == 0) report(p.status, LRKV_ERR_INDEX);
    for (int j = tid; j < D; j += kChunk) p.out[(static_cast<int64_t>(n) * p.Hq + m) * D + j] = 0.f;
    return;
  }
  const int pos = p.decode ? (len - 1) : (len - nq + qi);
  const int kv = m / (p.Hq / p.Hkv), half = D / 2;
  const bool bk = p.B_K != nullptr && a >= 0, bv = p.B_V != nullptr && a >= 0;
  const int loff = (p.lr_groups > 1 && a >= 0) ? a * R : 0;  // this adapter's low-rank group
  for (int j = tid; j < D; j += kChunk) qv[j] = p.q[(static_cast<int64_t>(n) * p.Hq + m) * D + j];
  for (int j = tid; j < D + R; j += kChunk) acc[j] = 0.f;
  __syncthreads();
  float m_run = -CUDART_INF_F, l_run = 0.f;
  const int64_t bstride = static_cast<int64_t>(p.Hkv) * D;
  for (int c0 = 0; c0 <= pos; c0 += kChunk) {
    // ---- scores of this chunk (one key per thread)
    const int t = c0 + tid;
    float s = -CUDART_INF_F;
    if (t <= pos) {
      const int blk = __ldg(p.block_tables + static_cast<int64_t>(c) * p.max_blocks + t / kBlock);
      if (blk >= 0 && blk < p.num_blocks) {
        const int row = t % kBlock;
        const float* kb = p.base_pool + (((static_cast<int64_t>(blk) * 2 + 0) * p.Hkv + kv) * kBlock + row) * D;
        const float* lk = p.lr_pool + ((static_cast<int64_t>(blk) * 2 + 0) * kBlock + row) * p.lrw + loff;
        float dotv = 0.f;
        for (int j = 0; j < half; ++j) {
          float x = 0.f, y = 0.f;
          if (bk) {
            const float* b = p.B_K + static_cast<int64_t>(a) * R * bstride + kv * D;
            for (int k = 0; k < R; ++k) {
              x = fmaf(lk[k], b[k * bstride + j], x);
              y = fmaf(lk[k], b[k * bstride + j + half], y);
            }
            const float2 cs = rope_cos_sin(t, p.freqs.hi[j], p.freqs.lo[j]);
            const float xr = x * cs.x - y * cs.y, yr = y * cs.x + x * cs.y;
            x = xr;
            y = yr;
          }
          dotv = fmaf(qv[j], kb[j] + x, dotv);
          dotv = fmaf(qv[j + half], kb[j + half] + y, dotv);
        }
        s = dotv * p.scale;
      } else if (m == 0) {
        report(p.status, LRKV_ERR_INDEX);
      }
    }
    // ---- chunk max, online update
    float mx = s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[wid] = mx;
    __syncthreads();
    mx = red[0];
    for (int w = 1; w < kChunk / 32; ++w) mx = fmaxf(mx, red[w]);
    const float mn = fmaxf(m_run, mx);
    const float al = (mn == -CUDART_INF_F) ? 1.f : expf(m_run - mn);
    const float pv = (mn == -CUDART_INF_F || s == -CUDART_INF_F) ? 0.f : expf(s - mn);
    sc[tid] = pv;
    float sum = pv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    __syncthreads();
    if (lane == 0) red[wid] = sum;
    __syncthreads();
    float csum = 0.f;
    for (int w = 0; w < kChunk / 32; ++w) csum += red[w];
    l_run = l_run * al + csum;
    m_run = mn;
    // ---- accumulate O (threads over columns)
    const int tn = min(kChunk, pos + 1 - c0);
    for (int j = tid; j < D + R; j += kChunk) {
      float v = acc[j] * al;
      if (j < D) {
        for (int i = 0; i < tn; ++i) {
          const int tt = c0 + i;
          const int blk = __ldg(p.block_tables + static_cast<int64_t>(c) * p.max_blocks + tt / kBlock);
          if (blk < 0 || blk >= p.num_blocks || sc[i] == 0.f) continue;
          v = fmaf(sc[i], p.base_pool[(((static_cast<int64_t>(blk) * 2 + 1) * p.Hkv + kv) * kBlock + tt % kBlock) * D + j], v);
        }
      } else if (bv) {
        for (int i = 0; i < tn; ++i) {
          const int tt = c0 + i;
          const int blk = __ldg(p.block_tables + static_cast<int64_t>(c) * p.max_blocks + tt / kBlock);
          if (blk < 0 || blk >= p.num_blocks || sc[i] == 0.f) continue;
          v = fmaf(sc[i], p.lr_pool[((static_cast<int64_t>(blk) * 2 + 1) * kBlock + tt % kBlock) * p.lrw + loff + (j - D)], v);
        }
      }
      acc[j] = v;
    }
    __syncthreads();
  }
  const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
  for (int j = tid; j < D; j += kChunk) {
    float v = acc[j];
    if (bv) {
      const float* b = p.B_V + static_cast<int64_t>(a) * R * bstride + kv * D + j;
      for (int k = 0; k < R; ++k) v = fmaf(acc[D + k], b[k * bstride], v);
    }
    p.out[(static_cast<int64_t>(n) * p.Hq + m) * D + j] = v * inv;
  }
}

lrkv_status attn_fp32(const lrkv_config& cfg, const float* q, const int32_t* row_start, int n_groups,
                      int max_rows, const int32_t* lens, int max_len, const int32_t* adapter_ids,
                      const int32_t* block_tables, int max_blocks, const void* base_pool,
                      const void* lr_pool, int64_t num_blocks, const void* B_K, const void* B_V,
                      int n_adapters, float scale, void* out, int32_t* status, int decode,
                      cudaStream_t stream) {
  if (n_groups == 0 || max_rows == 0) return LRKV_OK;
  Fp32AttnParams p{};
  p.q = q;
  p.row_start = row_start;
  p.lens = lens;
  p.adapter_ids = adapter_ids;
  p.block_tables = block_tables;
  p.base_pool = static_cast<const float*>(base_pool);
  p.lr_pool = static_cast<const float*>(lr_pool);
  p.B_K = static_cast<const float*>(B_K);
  p.B_V = static_cast<const float*>(B_V);
  p.out = static_cast<float*>(out);
  p.status = status;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks;
  p.max_len = max_len;
  p.Hq = cfg.n_q_heads;
  p.Hkv = cfg.n_kv_heads;
  p.D = cfg.head_dim;
  p.R = cfg.rank;
  p.lrw = lr_width(cfg);
  p.lr_groups = cfg.lr_groups;
  p.n_adapters = n_adapters;
  p.decode = decode;
  p.scale = scale;
  rope_freqs(cfg, &p.freqs);
  dim3 grid(n_groups, max_rows, cfg.n_q_heads);
  const int smem = (cfg.head_dim + kChunk + cfg.head_dim + cfg.rank + kChunk / 32 + 2) * 4;
  attn_fp32_kernel<<<grid, kChunk, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

}  // namespace

lrkv_status launch_append_fp32(const lrkv_config& cfg, const void* X_base, const void* X_lr, int T,
                               const int32_t* positions, const int32_t* seq_rows,
                               const int32_t* block_tables, int num_seqs, int max_blocks,
                               const void* W_cat, void* base_pool, void* lr_pool,
                               int64_t num_blocks, int32_t* status, cudaStream_t stream) {
  if (T == 0 || (X_base == nullptr && X_lr == nullptr)) return LRKV_OK;
  Fp32AppendParams p{};
  p.X_base = static_cast<const float*>(X_base);
  p.X_lr = static_cast<const float*>(X_lr);
  p.W = static_cast<const float*>(W_cat);
  p.positions = positions;
  p.seq_rows = seq_rows;
  p.block_tables = block_tables;
  p.base_pool = static_cast<float*>(base_pool);
  p.lr_pool = static_cast<float*>(lr_pool);
  p.status = status;
  p.num_blocks = num_blocks;
  p.h = cfg.hidden;
  p.Hkv = cfg.n_kv_heads;
  p.D = cfg.head_dim;
  p.R = cfg.rank;
  p.lrw = lr_width(cfg);
  p.num_seqs = num_seqs;
  p.max_blocks = max_blocks;
  rope_freqs(cfg, &p.freqs);
  const size_t smem = static_cast<size_t>(cfg.hidden) * 2 * 4;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(append_fp32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return LRKV_ERR_CUDA;
  append_fp32_kernel<<<T, 256, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

lrkv_status launch_decode_fp32(const lrkv_config& cfg, const DecodeArgs& a, int max_q_per_ctx,
                               cudaStream_t stream) {
  return attn_fp32(cfg, static_cast<const float*>(a.q), a.ctx_q_start, a.num_ctx, max_q_per_ctx,
                   a.ctx_lens, a.max_ctx_len, a.adapter_ids, a.block_tables, a.max_blocks,
                   a.base_pool, a.lr_pool, a.num_blocks, a.B_K, a.B_V, a.n_adapters, a.scale,
                   a.out, a.status, 1, stream);
}

lrkv_status launch_prefill_fp32(const lrkv_config& cfg, const PrefillArgs& a, cudaStream_t stream) {
  return attn_fp32(cfg, static_cast<const float*>(a.q), a.q_start, a.num_seqs, a.max_q_len,
                   a.seq_lens, a.max_seq_len, a.adapter_ids, a.block_tables, a.max_blocks,
                   a.base_pool, a.lr_pool, a.num_blocks, a.B_K, a.B_V, a.n_adapters, a.scale,
                   a.out, a.status, 0, stream);
}

}  // namespace lrkv
