// Cache append: one GEMM Y = X W_cat^T over the hidden size on the
// 5th-generation tensor cores, then an epilogue read straight from tensor
// memory that rotates the K columns (RoPE at each token's position), casts to
// bf16 and scatters every token row into its paged slot:
//   base_pool[blk][0][kv][row][:] = RoPE(Y_K),  base_pool[blk][1][kv][row][:] = Y_V,
//   lr_pool[blk][0][row][:] = Y_AK,              lr_pool[blk][1][row][:] = Y_AV.
// LRAgent (arXiv 2602.01053), Abstract: the base component is produced by the
// pretrained weights and the adapter component is kept low-rank; PReCache,
// Abstract: the low-rank cache is produced once, when a segment is first seen.
//
// Re-based appends (PReCache, Abstract and Figure 1, ReBaseShared): the base
// columns may come from one set of hidden states (the adapter-free pass) and
// the low-rank columns from another (the adapted pass), in one launch ("double
// batching", both paths together), or either part alone (a base-only re-base
// after an agent's turn, "lazy prefill"). The column tiles are laid out so
// that no tile mixes base and low-rank columns: base tiles of up to 256
// columns over [0, 2 Hkv d), then tiles of up to 256 over the 2 G r low-rank
// columns (G = lr_groups; PReCache, PreLRShared: every agent's own A in one
// GEMM when the segment is first processed).
//
// One CTA per (column tile, 128-token tile):
//   warp 0      TMA producer: X and W_cat k-slices (64 wide, 128-byte swizzle)
//               into a 4-stage mbarrier ring
//   warp 1      owns the tensor memory, issues tcgen05.mma (M = 128 tokens,
//               N = tile width, K = 16) into a fp32 accumulator in TMEM
//   warps 4-11  epilogue, two warpgroups splitting the tile's columns; thread
//               = token row = TMEM lane: tcgen05.ld, RoPE, bf16, 16-byte stores
// Every wait is bounded; a wait that gives up stores LRKV_ERR_TIMEOUT, raises
// the CTA's abort flag, and no copy or MMA is left in flight at exit.
#include <climits>

#include "lrkv_device.cuh"
#include "lrkv_internal.h"
#include "tcgen05.cuh"

namespace lrkv {
namespace {

constexpr int AM = 128;   // tokens per tile (MMA M, TMEM lanes)
constexpr int AN = 256;   // widest column tile (MMA N)
constexpr int AK = 64;    // k-slice: 64 bf16 = one 128-byte swizzle row
constexpr int NST = 4;    // pipeline stages
constexpr int kThreads = 384;
constexpr int A_BYTES = AM * AK * 2;            // 16 KB
constexpr int B_BYTES = AN * AK * 2;            // 32 KB
constexpr int STAGE = A_BYTES + B_BYTES;        // 48 KB
constexpr int OFF_BAR = NST * STAGE;
constexpr int SMEM_USED = OFF_BAR + 256;
constexpr int SMEM_TOTAL = SMEM_USED + 1024;    // + alignment slack
constexpr uint32_t kTmemCols = 256;
constexpr long long kWaitCycles = 1ll << 31;    // ~1 s: a wait this long has failed

enum : int { B_FULL = 0, B_EMPTY = NST, B_ACC = 2 * NST, B_DRAIN = 2 * NST + 1, B_COUNT = 2 * NST + 2 };

struct AppendParams {
  const int32_t* positions;
  const int32_t* seq_rows;
  const int32_t* block_tables;
  __nv_bfloat16* base_pool;
  __nv_bfloat16* lr_pool;
  int32_t* status;
  int64_t num_blocks;
  int T, h, Hkv, D, R, num_seqs, max_blocks;
  int kvc2;          // base columns: 2 * Hkv * D
  int lrw;           // low-rank row width: G * R (plane 0 = L_K, plane 1 = L_V)
  int n_base_tiles;  // base column tiles in the grid (0 when the base part is not written)
  int codec;         // 1: the base pool is compressed (q8_0 keys, rotated 3-bit values)
  float vthr[7];     // value-code thresholds (Lloyd-Max for N(0,1)), ascending
  RopeFreqs freqs;
};

// ------------------------------------------------------ compressed base pool
// One (block, kv head) chunk: Kq int8 [16][d] | Ks fp16 [16][d/32] |
// Vq u8 [16][3][d/8] | Vn fp32 [16] (PolyKV codec: the abstract printed at
// the end of the PReCache page).

// q8_0 of 32 values: scale s = max|x| / 127 (stored fp16), codes
// round(x / s) with ties away from zero; 32 bytes of codes.
__device__ __forceinline__ void q8_0_store(const float* x, int8_t* codes, __half* scale) {
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(x[e]));
  const float s = amax / 127.0f;
  const float inv = s > 0.f ? 1.0f / s : 0.f;
  uint32_t w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint32_t v = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float q = fminf(fmaxf(roundf(x[4 * k + e] * inv), -127.f), 127.f);
      v |= (static_cast<uint32_t>(static_cast<int>(q)) & 0xffu) << (8 * e);
    }
    w[k] = v;
  }
  *reinterpret_cast<uint4*>(codes) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(codes + 16) = make_uint4(w[4], w[5], w[6], w[7]);
  *scale = __float2half_rn(s);
}

// 3-bit code of u: the number of (ascending) thresholds below u, in three compares.
__device__ __forceinline__ uint32_t code3(float u, const float* t) {
  const bool b2 = t[3] < u;
  const bool b1 = (b2 ? t[5] : t[1]) < u;
  const float tl = b2 ? (b1 ? t[6] : t[4]) : (b1 ? t[2] : t[0]);
  return (b2 ? 4u : 0u) + (b1 ? 2u : 0u) + (tl < u ? 1u : 0u);
}

// Waits for an mbarrier phase; gives up (LRKV_ERR_TIMEOUT, false) after
// kWaitCycles, or early once another role has raised the abort flag.
__device__ __forceinline__ bool wait_ab(uint32_t bar, uint32_t parity, int32_t* st,
                                        const volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag != 0) return false;
    if (clock64() - t0 > kWaitCycles) {
      report(st, LRKV_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ uint4 pack8(const uint32_t* v) {
  return make_uint4(pack_bf16(__uint_as_float(v[0]), __uint_as_float(v[1])),
                    pack_bf16(__uint_as_float(v[2]), __uint_as_float(v[3])),
                    pack_bf16(__uint_as_float(v[4]), __uint_as_float(v[5])),
                    pack_bf16(__uint_as_float(v[6]), __uint_as_float(v[7])));
}

__global__ void __launch_bounds__(kThreads, 1)
    append_tc_kernel(const __grid_constant__ AppendParams p,
                     const __grid_constant__ CUtensorMap tm_xb,   // X of the base columns
                     const __grid_constant__ CUtensorMap tm_xl,   // X of the low-rank columns
                     const __grid_constant__ CUtensorMap tm_w) {  // W_cat [N][h]
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * B_COUNT + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool lr_tile = static_cast<int>(blockIdx.x) >= p.n_base_tiles;
  const int lt = static_cast<int>(blockIdx.x) - p.n_base_tiles;  // low-rank tile index
  const int n0 = lr_tile ? p.kvc2 + lt * AN : static_cast<int>(blockIdx.x) * AN;  // first output column
  const int width = lr_tile ? min(AN, 2 * p.lrw - lt * AN) : min(AN, p.kvc2 - n0);  // multiple of 16
  const int m0 = static_cast<int>(blockIdx.y) * AM;
  const int KT = p.h / AK;

  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tc::alloc(smem_u32(tmem_slot), kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // =========================================================== producer
    const CUtensorMap* xm = lr_tile ? &tm_xl : &tm_xb;
    if (lane == 0) {
      prefetch_tmap(xm);
      prefetch_tmap(&tm_w);
      bool ok = true;
      int issued = 0;
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % NST;
        if (kt >= NST && !wait_ab(bar(B_EMPTY + s), ((kt / NST) - 1) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t st = sbase + s * STAGE;
        mbar_arrive_expect_tx(bar(B_FULL + s), STAGE);
        tma_load_2d(st, xm, kt * AK, m0, bar(B_FULL + s));
        tma_load_2d(st + A_BYTES, &tm_w, kt * AK, n0, bar(B_FULL + s));
        ++issued;
      }
      if (!ok) {
        *abort_flag = 1;
        // no copy may still be landing when the CTA leaves
        for (int j = issued > NST ? issued - NST : 0; j < issued; ++j)
          wait_ab(bar(B_FULL + j % NST), (j / NST) & 1, p.status, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    const uint32_t idesc = tc::idesc_f16(AM, width, true, false, false);
    bool ok = true;
    int issued = 0;
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % NST;
      ok = __all_sync(0xffffffffu, wait_ab(bar(B_FULL + s), (kt / NST) & 1, p.status, abort_flag));
      if (!ok) break;
      tc::fence_after();
      if (tc::elect_one()) {
        const uint32_t st = sbase + s * STAGE;
        const uint64_t ad = tc::sdesc(st, 16, 1024, 2);
        const uint64_t bd = tc::sdesc(st + A_BYTES, 16, 1024, 2);
#pragma unroll
        for (int k = 0; k < AK / 16; ++k)  // 32 bytes along K per step, inside the swizzle row
          tc::mma_ss(tbase, ad + 2 * k, bd + 2 * k, idesc, (kt > 0 || k > 0) ? 1u : 0u);
        tc::commit(bar(B_EMPTY + s));
        if (kt == KT - 1) tc::commit(bar(B_ACC));
      }
      __syncwarp();
      ++issued;
    }
    if (!ok) {
      if (lane == 0) *abort_flag = 1;
      if (issued > 0) {
        if (tc::elect_one()) tc::commit(bar(B_DRAIN));
        __syncwarp();
        wait_ab(bar(B_DRAIN), 0, p.status, nullptr);
      }
    }
  } else if (warp >= 4) {
    // ============================================================== epilogue
    const int ew = warp - 4;
    const int grp = ew >> 2;  // column half [128 grp, 128 grp + 128) of the tile
    const int row = (ew & 3) * 32 + lane;
    const uint32_t tl = tbase + (static_cast<uint32_t>(32 * (ew & 3)) << 16);
    // this thread's token: block and row of its slot (skipped when out of range)
    const int t = m0 + row;
    int blk = -1, pos = 0;
    if (t < p.T) {
      const int s = __ldg(p.seq_rows + t);
      pos = __ldg(p.positions + t);
      if (s < 0 || s >= p.num_seqs || pos < 0 || pos >= p.max_blocks * kBlock) {
        if (blockIdx.x == 0 && grp == 0) report(p.status, LRKV_ERR_INDEX);
      } else {
        const int b = __ldg(p.block_tables + static_cast<int64_t>(s) * p.max_blocks + pos / kBlock);
        if (b < 0 || b >= p.num_blocks) {
          if (blockIdx.x == 0 && grp == 0) report(p.status, LRKV_ERR_INDEX);
        } else {
          blk = b;
        }
      }
    }
    const int slot_row = pos % kBlock;
    const int c_beg = grp * 128, c_end = min(width, c_beg + 128);
    const bool ok = __all_sync(0xffffffffu, wait_ab(bar(B_ACC), 0, p.status, abort_flag));
    if (ok && c_beg < c_end) {
      tc::fence_after();
      const int half = p.D / 2;
      const int kvc = p.kvc2 / 2;
      if (p.codec && !lr_tile) {
        // compressed base pool: one kv head's K or V columns per pass
        const int D = p.D, nb = p.D / 32;
        for (int c = c_beg; c < c_end; c += D) {
          const int n = n0 + c;
          const bool is_k = n < kvc;
          const int head = (is_k ? n : n - kvc) / D;
          uint8_t* chunk = blk >= 0 ? reinterpret_cast<uint8_t*>(p.base_pool) +
                                          (static_cast<int64_t>(blk) * p.Hkv + head) * (23 * D + 64)
                                    : nullptr;
          if (is_k) {
            // RoPE of the pairs (j, j + d/2), then q8_0 of each 32-dim block
            for (int j0 = 0; j0 < half; j0 += 32) {
              uint32_t lo[32], hi[32];
              tc::ld_x32(tl + c + j0, lo);
              tc::ld_x32(tl + c + j0 + half, hi);
              tc::wait_ld();
              float rl[32], rh[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const float2 cs = rope_cos_sin_fast(pos, p.freqs.hi[j0 + e], p.freqs.lo[j0 + e]);
                const float a = __uint_as_float(lo[e]), b = __uint_as_float(hi[e]);
                rl[e] = fmaf(a, cs.x, -(b * cs.y));
                rh[e] = fmaf(b, cs.x, a * cs.y);
              }
              if (chunk != nullptr) {
                int8_t* kq = reinterpret_cast<int8_t*>(chunk) + slot_row * D;
                __half* ks = reinterpret_cast<__half*>(chunk + 16 * D) + slot_row * nb;
                q8_0_store(rl, kq + j0, ks + j0 / 32);
                q8_0_store(rh, kq + j0 + half, ks + (j0 + half) / 32);
              }
            }
          } else {
            // ||v||, then (H v)_j / ||v|| per 32-wide group: H_d = H_{d/32} (x) H_32
            // (Sylvester), so group g is FWHT32 of sum_k (-1)^popc(g & k) v[32k ..]
            float ss = 0.f;
            for (int k = 0; k < nb; ++k) {
              uint32_t x[32];
              tc::ld_x32(tl + c + 32 * k, x);
              tc::wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) ss = fmaf(__uint_as_float(x[e]), __uint_as_float(x[e]), ss);
            }
            const float nrm = sqrtf(ss);
            const float inv = nrm > 0.f ? 1.0f / nrm : 0.f;
            uint32_t plane[3][4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              plane[0][g] = plane[1][g] = plane[2][g] = 0u;
              if (g < nb) {
                float z[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) z[e] = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  if (k < nb) {
                    uint32_t x[32];
                    tc::ld_x32(tl + c + 32 * k, x);
                    tc::wait_ld();
                    const bool neg = (__popc(g & k) & 1) != 0;
#pragma unroll
                    for (int e = 0; e < 32; ++e) z[e] += neg ? -__uint_as_float(x[e]) : __uint_as_float(x[e]);
                  }
                }
                fwht32(z);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                  const uint32_t q = code3(z[e] * inv, p.vthr);
                  plane[0][g] |= (q & 1u) << e;
                  plane[1][g] |= ((q >> 1) & 1u) << e;
                  plane[2][g] |= (q >> 2) << e;
                }
              }
            }
            if (chunk != nullptr) {
              uint32_t* vq = reinterpret_cast<uint32_t*>(chunk + 17 * D + slot_row * (3 * D / 8));
#pragma unroll
              for (int b = 0; b < 3; ++b)
#pragma unroll
                for (int g = 0; g < 4; ++g)
                  if (g < nb) vq[b * nb + g] = plane[b][g];
              reinterpret_cast<float*>(chunk + 23 * D)[slot_row] = nrm;
            }
          }
        }
      } else
      for (int c = c_beg; c < c_end; c += 16) {
        const int n = n0 + c;  // global output column of this 16-column group
        if (lr_tile) {
          uint32_t v[16];
          tc::ld_x16(tl + c, v);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int nn = n - p.kvc2 + 8 * e;  // low-rank column in [0, 2 G r)
            if (blk >= 0 && nn < 2 * p.lrw) {
              const int plane = nn / p.lrw, k0 = nn % p.lrw;
              *reinterpret_cast<uint4*>(p.lr_pool + ((static_cast<int64_t>(blk) * 2 + plane) * kBlock +
                                                     slot_row) * p.lrw + k0) = pack8(v + 8 * e);
            }
          }
        } else if (n < kvc) {
          // K: rotate the pair (j, j + d/2) of the head; the partner group sits
          // d/2 columns further in the same tile half (heads are d-aligned)
          const int j0 = n % p.D;
          if (j0 >= half) continue;  // handled with its low half
          uint32_t lo[16], hi[16];
          tc::ld_x16(tl + c, lo);
          tc::ld_x16(tl + c + half, hi);
          tc::wait_ld();
          uint32_t rl[16], rh[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 cs = rope_cos_sin_fast(pos, p.freqs.hi[j0 + e], p.freqs.lo[j0 + e]);
            const float a = __uint_as_float(lo[e]), b = __uint_as_float(hi[e]);
            rl[e] = __float_as_uint(fmaf(a, cs.x, -(b * cs.y)));
            rh[e] = __float_as_uint(fmaf(b, cs.x, a * cs.y));
          }
          if (blk >= 0) {
            __nv_bfloat16* dst = p.base_pool + (((static_cast<int64_t>(blk) * 2 + 0) * p.Hkv + n / p.D) * kBlock +
                                                slot_row) * p.D + j0;
            *reinterpret_cast<uint4*>(dst) = pack8(rl);
            *reinterpret_cast<uint4*>(dst + 8) = pack8(rl + 8);
            *reinterpret_cast<uint4*>(dst + half) = pack8(rh);
            *reinterpret_cast<uint4*>(dst + half + 8) = pack8(rh + 8);
          }
        } else {
          // V: stored as computed
          uint32_t v[16];
          tc::ld_x16(tl + c, v);
          tc::wait_ld();
          if (blk >= 0) {
            const int nn = n - kvc;
            __nv_bfloat16* dst = p.base_pool + (((static_cast<int64_t>(blk) * 2 + 1) * p.Hkv + nn / p.D) * kBlock +
                                                slot_row) * p.D + nn % p.D;
            *reinterpret_cast<uint4*>(dst) = pack8(v);
            *reinterpret_cast<uint4*>(dst + 8) = pack8(v + 8);
          }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tbase, kTmemCols);
  }
}

// Tensor map over a row-major bf16 matrix [rows][h], box {64, box_rows},
// 128-byte swizzle (one box row = one swizzle row).
bool make_kmajor_map(const void* base, int64_t rows, int h, int box_rows, CUtensorMap* map) {
  return make_bf16_2d_map(base, h, rows, static_cast<int64_t>(h) * 2, AK, box_rows, 128, map);
}

}  // namespace

lrkv_status launch_append_bf16(const lrkv_config& cfg, const void* X_base, const void* X_lr, int T,
                               const int32_t* positions, const int32_t* seq_rows,
                               const int32_t* block_tables, int num_seqs, int max_blocks,
                               const void* W_cat, void* base_pool, void* lr_pool,
                               int64_t num_blocks, int32_t* status, cudaStream_t stream) {
  if (T == 0 || (X_base == nullptr && X_lr == nullptr)) return LRKV_OK;
  AppendParams p{};
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
  p.num_seqs = num_seqs;
  p.max_blocks = max_blocks;
  p.kvc2 = 2 * cfg.n_kv_heads * cfg.head_dim;
  p.lrw = lr_width(cfg);
  p.n_base_tiles = X_base != nullptr ? (p.kvc2 + AN - 1) / AN : 0;
  p.codec = cfg.kv_codec == LRKV_CODEC_POLYKV ? 1 : 0;
  for (int k = 0; k < 7; ++k) p.vthr[k] = polykv_codec().threshold[k];
  const int n_lr_tiles = X_lr != nullptr ? (2 * p.lrw + AN - 1) / AN : 0;
  rope_freqs(cfg, &p.freqs);
  const int64_t N = p.kvc2 + 2 * p.lrw;
  CUtensorMap xb, xl, wm;
  const void* xb_src = X_base != nullptr ? X_base : X_lr;
  const void* xl_src = X_lr != nullptr ? X_lr : X_base;
  if (!make_kmajor_map(xb_src, T, cfg.hidden, AM, &xb) || !make_kmajor_map(xl_src, T, cfg.hidden, AM, &xl) ||
      !make_kmajor_map(W_cat, N, cfg.hidden, AN, &wm))
    return LRKV_ERR_CUDA;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(append_tc_kernel), SMEM_TOTAL)) return LRKV_ERR_CUDA;
  dim3 grid(p.n_base_tiles + n_lr_tiles, (T + AM - 1) / AM);
  append_tc_kernel<<<grid, kThreads, SMEM_TOTAL, stream>>>(p, xb, xl, wm);
  return cudaGetLastError() == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

}  // namespace lrkv
