// Cache append: one GEMM Y = X W_cat^T over the hidden size, then a fused
// epilogue that rotates the K columns (RoPE at each token's position), casts
// to bf16 and scatters every token row into its paged slot:
//   base_pool[blk][0][kv][row][:] = RoPE(Y_K),  base_pool[blk][1][kv][row][:] = Y_V,
//   lr_pool[blk][0][row][:] = Y_AK,              lr_pool[blk][1][row][:] = Y_AV.
// LRAgent (arXiv 2602.01053), Abstract: the base component is produced by the
// pretrained weights and the adapter component is kept low-rank; PReCache,
// Abstract: the low-rank cache is produced once, when a segment is first seen.
//
// GEMM: 128x128x32 CTA tiles, 8 warps of 64x32, legacy warp MMAs
// (m16n8k16 bf16, fp32 accumulate), 4-stage cp.async pipeline with an XOR
// swizzle so every ldmatrix is conflict-free.
#include <algorithm>

#include "lrkv_device.cuh"
#include "lrkv_internal.h"

namespace lrkv {
namespace {

constexpr int BM = 128, BN = 128, BK = 32, NSTAGE = 4, NTHR = 256;
constexpr int TILE_BYTES = BM * BK * 2;  // 8 KB per operand per stage
constexpr int EPI_PITCH = BN + 4;        // floats
constexpr int SMEM_PIPE = NSTAGE * 2 * TILE_BYTES;
constexpr int SMEM_EPI = BM * EPI_PITCH * 4;
constexpr int SMEM_ROWS = BM * 16;  // per-row slot info
constexpr int SMEM_TOTAL = (SMEM_PIPE > SMEM_EPI ? SMEM_PIPE : SMEM_EPI) + SMEM_ROWS;

struct AppendParams {
  const __nv_bfloat16* X;
  const __nv_bfloat16* W;  // [N][h]
  const int32_t* positions;
  const int32_t* seq_rows;
  const int32_t* block_tables;
  __nv_bfloat16* base_pool;
  __nv_bfloat16* lr_pool;
  int32_t* status;
  int64_t num_blocks;
  int T, h, N, Hkv, D, R, num_seqs, max_blocks;
  RopeFreqs freqs;
};

// 64-byte rows of 4 16-byte chunks; chunk index XOR (row / 2) % 4.
__device__ __forceinline__ uint32_t sw_off(int row, int chunk) {
  return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  const int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(NTHR) append_gemm_kernel(const __grid_constant__ AppendParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  int* rowinfo = reinterpret_cast<int*>(smem + (SMEM_PIPE > SMEM_EPI ? SMEM_PIPE : SMEM_EPI));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int wm = warp >> 2, wn = warp & 3;  // 2 x 4 warps, 64 x 32 each

  auto load_stage = [&](int s, int k0) {
    const uint32_t xa = sb + s * 2 * TILE_BYTES, wa = xa + TILE_BYTES;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int v = tid + i * NTHR;  // 512 16-byte vectors per operand
      const int row = v >> 2, ch = v & 3;
      const int xr = m0 + row, wr = n0 + row;
      const bool px = xr < p.T, pw = wr < p.N;
      const __nv_bfloat16* xs = p.X + static_cast<int64_t>(px ? xr : 0) * p.h + k0 + ch * 8;
      const __nv_bfloat16* ws = p.W + static_cast<int64_t>(pw ? wr : 0) * p.h + k0 + ch * 8;
      cp_async16(xa + sw_off(row, ch), xs, px);
      cp_async16(wa + sw_off(row, ch), ws, pw);
    }
  };

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;

  const int KT = p.h / BK;
#pragma unroll
  for (int s = 0; s < NSTAGE - 1; ++s) {
    if (s < KT) load_stage(s, s * BK);
    cp_commit();
  }
  for (int kt = 0; kt < KT; ++kt) {
    cp_wait<NSTAGE - 2>();
    __syncthreads();
    const int nk = kt + NSTAGE - 1;
    if (nk < KT) load_stage(nk % NSTAGE, nk * BK);
    cp_commit();
    const int s = kt % NSTAGE;
    const uint32_t xa = sb + s * 2 * TILE_BYTES, wa = xa + TILE_BYTES;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {  // two k16 steps per BK = 32
      uint32_t af[4][4], bfr[2][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int mi = lane >> 3;
        const int row = wm * 64 + mt * 16 + (lane & 7) + (mi & 1) * 8;
        const int ch = kk * 2 + (mi >> 1);
        ldsm_x4(af[mt], xa + sw_off(row, ch));
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        // W rows are output columns (B "col" operand): non-transposed ldmatrix
        const int mi = lane >> 3;
        const int row = wn * 32 + np * 16 + (lane & 7) + (mi >> 1) * 8;
        const int ch = kk * 2 + (mi & 1);
        ldsm_x4(bfr[np], wa + sw_off(row, ch));
      }
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          mma16816(acc[mt][nt], af[mt], bfr[nt >> 1][(nt & 1) * 2], bfr[nt >> 1][(nt & 1) * 2 + 1]);
    }
  }
  cp_wait<0>();
  __syncthreads();

  // ---- stage the fp32 tile and the per-row slot info
  float* ep = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int r = wm * 64 + mt * 16 + (lane >> 2);
      const int c = wn * 32 + nt * 8 + (lane & 3) * 2;
      ep[r * EPI_PITCH + c] = acc[mt][nt][0];
      ep[r * EPI_PITCH + c + 1] = acc[mt][nt][1];
      ep[(r + 8) * EPI_PITCH + c] = acc[mt][nt][2];
      ep[(r + 8) * EPI_PITCH + c + 1] = acc[mt][nt][3];
    }
  if (tid < BM) {
    const int t = m0 + tid;
    int blk = -1, pos = 0;
    if (t < p.T) {
      const int s = __ldg(p.seq_rows + t);
      pos = __ldg(p.positions + t);
      if (s < 0 || s >= p.num_seqs || pos < 0 || pos >= p.max_blocks * kBlock) {
        if (blockIdx.x == 0) report(p.status, LRKV_ERR_INDEX);
      } else {
        const int b = __ldg(p.block_tables + static_cast<int64_t>(s) * p.max_blocks + pos / kBlock);
        if (b < 0 || b >= p.num_blocks) {
          if (blockIdx.x == 0) report(p.status, LRKV_ERR_INDEX);
        } else {
          blk = b;
        }
      }
    }
    rowinfo[tid * 2] = blk;
    rowinfo[tid * 2 + 1] = pos;
  }
  __syncthreads();

  // ---- rotate / cast / scatter, 8 columns per task
  const int kvc = p.Hkv * p.D;
  const int half = p.D / 2;
  for (int task = tid; task < BM * (BN / 8); task += NTHR) {
    const int r = task / (BN / 8), c8 = (task % (BN / 8)) * 8;
    const int n = n0 + c8;
    const int blk = rowinfo[r * 2];
    if (n >= p.N || blk < 0) continue;
    const int pos = rowinfo[r * 2 + 1];
    const float* src = ep + r * EPI_PITCH + c8;
    float v[8];
    __nv_bfloat16* dst;
    if (n < kvc) {  // K: rotate with the partner half of the same head
      const int kv = n / p.D, j0 = n % p.D;
      const bool lo = j0 < half;
      const float* partner = src + (lo ? half : -half);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int jj = (j0 + e) % half;
        const float2 cs = rope_cos_sin(pos, p.freqs.hi[jj], p.freqs.lo[jj]);
        v[e] = lo ? (src[e] * cs.x - partner[e] * cs.y) : (src[e] * cs.x + partner[e] * cs.y);
      }
      dst = p.base_pool + (((static_cast<int64_t>(blk) * 2 + 0) * p.Hkv + kv) * kBlock + pos % kBlock) * p.D + j0;
    } else if (n < 2 * kvc) {
      const int nn = n - kvc, kv = nn / p.D, j0 = nn % p.D;
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = src[e];
      dst = p.base_pool + (((static_cast<int64_t>(blk) * 2 + 1) * p.Hkv + kv) * kBlock + pos % kBlock) * p.D + j0;
    } else {
      const int nn = n - 2 * kvc;  // [0, 2R)
      const int plane = nn / p.R, k0 = nn % p.R;
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = src[e];
      dst = p.lr_pool + ((static_cast<int64_t>(blk) * 2 + plane) * kBlock + pos % kBlock) * p.R + k0;
    }
    uint4 pk;
    pk.x = pack_bf16(v[0], v[1]);
    pk.y = pack_bf16(v[2], v[3]);
    pk.z = pack_bf16(v[4], v[5]);
    pk.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4*>(dst) = pk;
  }
}

}  // namespace

lrkv_status launch_append_bf16(const lrkv_config& cfg, const void* X, int T,
                               const int32_t* positions, const int32_t* seq_rows,
                               const int32_t* block_tables, int num_seqs, int max_blocks,
                               const void* W_cat, void* base_pool, void* lr_pool,
                               int64_t num_blocks, int32_t* status, cudaStream_t stream) {
  if (T == 0) return LRKV_OK;
  AppendParams p{};
  p.X = static_cast<const __nv_bfloat16*>(X);
  p.W = static_cast<const __nv_bfloat16*>(W_cat);
  p.positions = positions;
  p.seq_rows = seq_rows;
  p.block_tables = block_tables;
  p.base_pool = static_cast<__nv_bfloat16*>(base_pool);
  p.lr_pool = static_cast<__nv_bfloat16*>(lr_pool);
  p.status = status;
  p.num_blocks = num_blocks;
  p.T = T;
  p.h = cfg.hidden;
  p.Hkv = cfg.n_kv_heads;
  p.D = cfg.head_dim;
  p.R = cfg.rank;
  p.N = 2 * cfg.n_kv_heads * cfg.head_dim + 2 * cfg.rank;
  p.num_seqs = num_seqs;
  p.max_blocks = max_blocks;
  rope_freqs(cfg, &p.freqs);
  if (!ensure_smem_attr(reinterpret_cast<const void*>(append_gemm_kernel), SMEM_TOTAL)) return LRKV_ERR_CUDA;
  dim3 grid((p.N + BN - 1) / BN, (T + BM - 1) / BM);
  append_gemm_kernel<<<grid, NTHR, SMEM_TOTAL, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

}  // namespace lrkv
