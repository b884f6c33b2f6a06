// Causal prefill attention over the paged base + shared-A low-rank cache (bf16).
//
// LRAgent (arXiv 2602.01053), Abstract (Flash-LoRA-Attention): each agent's
// K adapter term L_K B_K is rebuilt per key tile on chip, rotated and added to
// K_base; the V term is reordered as (P L_V) B_V. PReCache, Abstract: a new
// turn attends over the context cached by earlier agents plus its own chunk.
//
// One CTA per (sequence, kv head, tile of 64 query rows); rows are
// (query, head-in-group) pairs so the g query heads sharing a kv head share
// every key tile. A producer warp streams 64-key tiles (4 paged blocks: K/V
// halves and L_K/L_V) with 2-D TMA copies into an mbarrier ring; each of the
// four consumer warps rebuilds one block of K_a = K_base + RoPE(L_K B_K,a)
// into a shared, swizzled fp16 tile, then all four compute S = Q K_a^T (fp16
// operands, fp32 accumulation), the causal
// mask (bottom-right aligned), the online softmax, O += P V_base and
// O_lr += P L_V with legacy warp MMAs. The epilogue applies O_lr B_V,a and 1/l.
#include <math_constants.h>

#include <algorithm>

#include "lrkv_device.cuh"
#include "lrkv_internal.h"

namespace lrkv {
namespace {

constexpr int kNW = 4;
constexpr int kThreads = (kNW + 1) * 32;
constexpr int BMQ = 64;   // query rows per CTA (16 per consumer warp)
constexpr int BKEY = 64;  // keys per tile (kNW blocks)
constexpr int kSmemLimit = 227 * 1024;

struct PrefillParams {
  const __nv_bfloat16* q;
  const int32_t* q_start;
  const int32_t* seq_lens;
  const int32_t* adapter_ids;
  const int32_t* block_tables;
  const __nv_bfloat16* B_K;
  const __nv_bfloat16* B_V;
  __nv_bfloat16* out;
  int32_t* status;
  int64_t num_blocks;
  int num_seqs, max_blocks, max_seq_len, n_adapters, Hq, Hkv, g, nstage;
  int has_bk, has_bv;
  float scale_log2;
  RopeFreqs freqs;
};

struct PLayout {
  int kv_tile, lr_tile, stage, ki_buf, bk_pitch, d_pitch;
  int off_ki, off_bk, off_bv, off_olr, off_dtab, off_btab, off_freq, off_misc, off_bar, total;
  __host__ __device__ static PLayout make(int D, int R, int nstage) {
    PLayout L;
    L.kv_tile = 16 * D * 2;
    L.lr_tile = 16 * R * 2;
    L.stage = kNW * (2 * L.kv_tile + 2 * L.lr_tile);
    L.ki_buf = BKEY * D * 2;
    L.bk_pitch = (D + 8) * 2;
    L.d_pitch = (D / 2) * 8 + 64;
    int o = nstage * L.stage;
    L.off_ki = o;   o += 2 * L.ki_buf;
    L.off_bk = o;   o += R * L.bk_pitch;
    o = (o + 15) & ~15;
    L.off_bv = o;   o += R * D * 4;
    L.off_olr = o;  o += BMQ * (R + 4) * 4;
    L.off_dtab = o; o += 16 * L.d_pitch;
    L.off_btab = o; o += kNW * (D / 2) * 8;
    L.off_freq = o; o += 2 * 64 * 4;
    L.off_misc = o; o += 64;
    o = (o + 7) & ~7;
    L.off_bar = o;  o += 2 * nstage * 8;
    L.total = o + 1024;
    return L;
  }
};

template <int D, int R>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p,
                   const __grid_constant__ CUtensorMap tm_base,
                   const __grid_constant__ CUtensorMap tm_lr) {
  constexpr int HALF = D / 2;
  constexpr int NCH = D / 32;
  constexpr int NKS = D / 16;
  constexpr int NRT = R >= 16 ? R / 16 : 1;
  constexpr int NLR = R / 8;
  constexpr int LR_RB = R * 2;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const PLayout L = PLayout::make(D, R, p.nstage);
  const uint32_t sbase = smem_u32(smem);
  float2* dtab = reinterpret_cast<float2*>(smem + L.off_dtab);
  float* freq = reinterpret_cast<float*>(smem + L.off_freq);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.off_misc);
  int* stage_mask = reinterpret_cast<int*>(smem + L.off_misc + 16);
  const uint32_t bar_full = sbase + L.off_bar;
  const uint32_t bar_empty = bar_full + 8 * p.nstage;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, c4 = lane & 3;
  const int s = blockIdx.z, head = blockIdx.y, tile = blockIdx.x;

  const int qs = __ldg(p.q_start + s), qe = __ldg(p.q_start + s + 1);
  const int q_len = qe - qs;
  int Ls = __ldg(p.seq_lens + s);
  const int g = p.g;
  const int row0 = tile * BMQ;             // first (query, head) row of this CTA
  if (row0 >= q_len * g) return;           // whole CTA beyond this sequence's chunk
  if (Ls < q_len || Ls > p.max_seq_len) {  // inconsistent lengths: skip, report
    if (tid == 0) report(p.status, LRKV_ERR_INDEX);
    return;
  }
  int adapter = __ldg(p.adapter_ids + s);
  if (adapter < -1 || adapter >= p.n_adapters) {
    if (tid == 0) report(p.status, LRKV_ERR_INDEX);
    adapter = -1;
  }
  const bool rebuild = p.has_bk && adapter >= 0;
  const bool use_lr = p.has_bv && adapter >= 0;
  const int k_first = row0 / g;
  const int k_last = min(q_len, (row0 + BMQ + g - 1) / g) - 1;
  const int pos_min = Ls - q_len + k_first;
  const int pos_max = Ls - q_len + k_last;
  const int n_tiles = (pos_max + BKEY) / BKEY;  // keys 0 .. pos_max

  // ---- prologue
  if (tid < HALF) {
    freq[tid] = p.freqs.hi[tid];
    freq[64 + tid] = p.freqs.lo[tid];
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < p.nstage; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, kNW);
    }
    mbar_fence_init();
  }
  __syncthreads();
  for (int i = tid; i < 16 * HALF; i += kThreads) {
    const int dl = i / HALF, j = i % HALF;
    *reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(dtab) + dl * L.d_pitch + j * 8) =
        rope_cos_sin(dl, freq[j], freq[64 + j]);
  }
  if (rebuild) {
    const __nv_bfloat16* src = p.B_K + static_cast<int64_t>(adapter) * R * p.Hkv * D + head * D;
    for (int i = tid; i < R * (D / 8); i += kThreads) {
      const int k = i / (D / 8), v = i % (D / 8);
      *reinterpret_cast<uint4*>(smem + L.off_bk + k * L.bk_pitch + v * 16) =
          __ldg(reinterpret_cast<const uint4*>(src + static_cast<int64_t>(k) * p.Hkv * D) + v);
    }
  }
  if (use_lr) {
    const __nv_bfloat16* src = p.B_V + static_cast<int64_t>(adapter) * R * p.Hkv * D + head * D;
    float* bv = reinterpret_cast<float*>(smem + L.off_bv);
    for (int i = tid; i < R * D; i += kThreads)
      bv[i] = __bfloat162float(src[static_cast<int64_t>(i / D) * p.Hkv * D + i % D]);
  }
  __syncthreads();

  const int nblk_seq = (Ls + kBlock - 1) / kBlock;

  // ======================================================== producer warp
  if (warp == kNW) {
    if (lane == 0) {
      prefetch_tmap(&tm_base);
      prefetch_tmap(&tm_lr);
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      for (int kt = 0; kt < n_tiles; ++kt) {
        if (*abort_flag || !mbar_wait(bar_empty + 8 * stage, phase ^ 1, p.status)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        int mask = 0, blks[kNW];
        uint32_t bytes = 0;
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
          blks[w] = -1;
          const int b = kt * kNW + w;
          if (b >= nblk_seq) continue;
          const int blk = __ldg(p.block_tables + static_cast<int64_t>(s) * p.max_blocks + b);
          if (blk < 0 || blk >= p.num_blocks) {
            report(p.status, LRKV_ERR_INDEX);
            continue;
          }
          blks[w] = blk;
          mask |= 1 << w;
          bytes += 2 * L.kv_tile + (rebuild ? L.lr_tile : 0) + (use_lr ? L.lr_tile : 0);
        }
        stage_mask[stage] = mask;
        const uint32_t fb = bar_full + 8 * stage;
        mbar_arrive_expect_tx(fb, bytes);
        issued |= 1u << stage;
        const uint32_t st = sbase + stage * L.stage;
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
          if (blks[w] < 0) continue;
          const int blk = blks[w];
          const int yk = ((blk * 2 + 0) * p.Hkv + head) * kBlock;
          const int yv = ((blk * 2 + 1) * p.Hkv + head) * kBlock;
          const uint32_t kt_s = st + w * L.kv_tile;
          const uint32_t vt_s = st + kNW * L.kv_tile + w * L.kv_tile;
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_2d(kt_s + h * 2048, &tm_base, 64 * h, yk, fb);
            tma_load_2d(vt_s + h * 2048, &tm_base, 64 * h, yv, fb);
          }
          const uint32_t lk = st + 2 * kNW * L.kv_tile + w * L.lr_tile;
          if (rebuild) tma_load_2d(lk, &tm_lr, 0, (blk * 2 + 0) * kBlock, fb);
          if (use_lr) tma_load_2d(lk + kNW * L.lr_tile, &tm_lr, 0, (blk * 2 + 1) * kBlock, fb);
        }
        if (++stage == p.nstage) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        for (int i = 0; i < p.nstage; ++i)
          if (issued >> i & 1) mbar_wait(bar_full + 8 * i, (i < stage) ? phase : (phase ^ 1), nullptr, 1u << 16);
      }
    }
    return;
  }

  // ======================================================= consumer warps
  float2* btab = reinterpret_cast<float2*>(smem + L.off_btab) + warp * HALF;
  // Q A fragments: rows (16*warp + g8, + 8), straight from global
  uint32_t qa[NKS][4];
  int rpos[2];
  bool rvalid[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = row0 + 16 * warp + g8 + 8 * h;
    const int k = r / g;
    rvalid[h] = k < q_len;
    rpos[h] = Ls - q_len + (rvalid[h] ? k : 0);
    const __nv_bfloat16* qrow =
        p.q + (static_cast<int64_t>(qs + (rvalid[h] ? k : 0)) * p.Hq + head * g + r % g) * D;
#pragma unroll
    for (int ks = 0; ks < NKS; ++ks) {
      qa[ks][h] = rvalid[h] ? bf16x2_to_f16x2(__ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c4))) : 0u;
      qa[ks][h + 2] = rvalid[h] ? bf16x2_to_f16x2(__ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * c4))) : 0u;
    }
  }
  float O[D / 8][4];
  float Olr[NLR][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
#pragma unroll
  for (int i = 0; i < NLR; ++i) Olr[i][0] = Olr[i][1] = Olr[i][2] = Olr[i][3] = 0.f;
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F}, l_run[2] = {0.f, 0.f};

  int stage = 0;
  uint32_t phase = 0;
  for (int kt = 0; kt < n_tiles; ++kt) {
    // every wait result is made warp-uniform before any warp-collective use
    bool ok = !__shfl_sync(0xffffffffu, *abort_flag, 0);
    if (ok) ok = mbar_wait(bar_full + 8 * stage, phase, p.status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) *abort_flag = 1;
    const int mask = ok ? stage_mask[stage] : 0;
    const uint32_t st = sbase + stage * L.stage;
    const uint32_t ki = sbase + L.off_ki + (kt & 1) * L.ki_buf;

    // ---- this warp's block: K_a = K_base + RoPE(L_K B_K) -> ki (swizzled)
    {
      const int b = kt * kNW + warp;
      const int t0 = b * kBlock;
      const uint32_t kts = st + warp * L.kv_tile;
      const uint32_t lkt = st + 2 * kNW * L.kv_tile + warp * L.lr_tile;
      const bool have = (mask >> warp) & 1;
      // Rows past the sequence end may hold stale pool memory: zero their V and
      // L_V rows so that P = 0 there cannot meet a NaN in the PV products.
      if (have && t0 + kBlock > Ls) {
        const uint32_t vts = st + kNW * L.kv_tile + warp * L.kv_tile;
        const uint32_t lvts = lkt + kNW * L.lr_tile;
        const int r0 = Ls - t0;
        for (int i = lane; i < (kBlock - r0) * (D / 8); i += 32) {
          const int r = r0 + i / (D / 8), v = i % (D / 8);
          const uint32_t a = vts + (v / 8) * 2048 + r * 128 + (v % 8) * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(a), "r"(0u) : "memory");
        }
        for (int i = lane; i < (kBlock - r0) * (R / 8); i += 32) {
          const int r = r0 + i / (R / 8), v = i % (R / 8);
          const uint32_t a = lvts + r * LR_RB + v * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(a), "r"(0u) : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        __syncwarp();
      }
      if (rebuild && have) {
        for (int j = lane; j < HALF; j += 32) btab[j] = rope_cos_sin(t0, freq[j], freq[64 + j]);
        __syncwarp();
      }
      uint32_t alk[NRT][4];
      if (rebuild && have) {
        if constexpr (R >= 16) {
#pragma unroll
          for (int ks = 0; ks < NRT; ++ks) {
            const int mi = lane >> 3;
            ldsm_x4(alk[ks], lkt + swz<LR_RB>((lane & 7) + (mi & 1) * 8, (2 * ks + (mi >> 1)) * 16));
          }
        } else {
          uint32_t t2[2];
          ldsm_x2(t2, lkt + swz<LR_RB>((lane & 7) + ((lane >> 3) & 1) * 8, 0));
          alk[0][0] = t2[0];
          alk[0][1] = t2[1];
          alk[0][2] = alk[0][3] = 0u;
        }
      }
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        uint32_t kbv[2][2][2];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int tk = 0; tk < 2; ++tk) {
              const int j = 16 * cc + 8 * n + 2 * c4 + h * HALF;
              uint32_t v = 0u;
              if (have) {
                const uint32_t addr = kts + (j / 64) * 2048 + swz<128>(g8 + 8 * tk, (j % 64) * 2);
                asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
              }
              kbv[n][h][tk] = v;
            }
        uint32_t outv[2][2][2];
        if (rebuild && have) {
          float2 cs[2][2][2];
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            const int j = 16 * cc + 8 * n + 2 * c4;
            const float4 bq = *reinterpret_cast<const float4*>(btab + j);
#pragma unroll
            for (int tk = 0; tk < 2; ++tk) {
              const float4 dq = *reinterpret_cast<const float4*>(
                  reinterpret_cast<const uint8_t*>(dtab) + (g8 + 8 * tk) * L.d_pitch + j * 8);
              cs[tk][n][0] = make_float2(bq.x * dq.x - bq.y * dq.y, bq.y * dq.x + bq.x * dq.y);
              cs[tk][n][1] = make_float2(bq.z * dq.z - bq.w * dq.w, bq.w * dq.z + bq.z * dq.w);
            }
          }
          float y[4][4];
#pragma unroll
          for (int i = 0; i < 4; ++i) y[i][0] = y[i][1] = y[i][2] = y[i][3] = 0.f;
          const uint32_t bk = sbase + L.off_bk;
          if constexpr (R >= 16) {
#pragma unroll
            for (int ks = 0; ks < NRT; ++ks)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int mi = lane >> 3;
                const int krow = 16 * ks + (lane & 7) + (mi & 1) * 8;
                const int ncol = 16 * cc + h * HALF + (mi >> 1) * 8;
                uint32_t bb[4];
                ldsm_x4_t(bb, bk + krow * L.bk_pitch + ncol * 2);
                mma16816(y[2 * h + 0], alk[ks], bb[0], bb[1]);
                mma16816(y[2 * h + 1], alk[ks], bb[2], bb[3]);
              }
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int ncol = 16 * cc + h * HALF + ((lane >> 3) & 1) * 8;
              uint32_t bb[2];
              ldsm_x2_t(bb, bk + (lane & 7) * L.bk_pitch + ncol * 2);
              mma1688(y[2 * h + 0], alk[0][0], alk[0][1], bb[0]);
              mma1688(y[2 * h + 1], alk[0][0], alk[0][1], bb[1]);
            }
          }
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int tk = 0; tk < 2; ++tk) {
              float lo2[2], hi2[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int i = 2 * tk + e;
                const float x = y[n][i], yy = y[n + 2][i];
                const float c = cs[tk][n][e].x, sn = cs[tk][n][e].y;
                const float blo = e ? bf16_hi(kbv[n][0][tk]) : bf16_lo(kbv[n][0][tk]);
                const float bhi = e ? bf16_hi(kbv[n][1][tk]) : bf16_lo(kbv[n][1][tk]);
                lo2[e] = fmaf(x, c, fmaf(-yy, sn, blo));
                hi2[e] = fmaf(yy, c, fmaf(x, sn, bhi));
              }
              outv[n][0][tk] = pack_f16(lo2[0], lo2[1]);
              outv[n][1][tk] = pack_f16(hi2[0], hi2[1]);
            }
        } else {
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int tk = 0; tk < 2; ++tk) outv[n][h][tk] = bf16x2_to_f16x2(kbv[n][h][tk]);
        }
        // store into ki: [D/64 halves][64 keys][64 dims], 128-byte swizzle
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int tk = 0; tk < 2; ++tk) {
              const int j = 16 * cc + 8 * n + 2 * c4 + h * HALF;
              const int key = 16 * warp + g8 + 8 * tk;
              const uint32_t addr = ki + (j / 64) * (BKEY * 128) + swz<128>(key, (j % 64) * 2);
              asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(addr), "r"(outv[n][h][tk]) : "memory");
            }
      }
    }
    named_bar_sync(1, kNW * 32);

    // ---- S = Q K_a^T for this warp's 16 rows x 64 keys
    float sacc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < NKS; ++ks)
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int mi = lane >> 3;
        const int key = 16 * np + (lane & 7) + (mi >> 1) * 8;
        const int dim = 16 * ks + (mi & 1) * 8;
        uint32_t bb[4];
        ldsm_x4(bb, ki + (dim / 64) * (BKEY * 128) + swz<128>(key, (dim % 64) * 2));
        mma16816_f16(sacc[2 * np], qa[ks], bb[0], bb[1]);
        mma16816_f16(sacc[2 * np + 1], qa[ks], bb[2], bb[3]);
      }
    // ---- mask, online softmax (rows g8, g8 + 8)
    const int key0 = kt * BKEY;
    const bool need_mask = key0 + BKEY - 1 > pos_min;
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key0 + 8 * nt + 2 * c4 + e;
          const int blkw = (8 * nt + 2 * c4 + e) >> 4;
          float v = sacc[nt][2 * h + e] * p.scale_log2;
          const bool vis = ((mask >> blkw) & 1) && (!need_mask || key <= rpos[h]) && rvalid[h];
          v = vis ? v : -CUDART_INF_F;
          sacc[nt][2 * h + e] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mn = fmaxf(m_run[h], mx);
      float sum = 0.f;
      if (mn == -CUDART_INF_F) {
        alpha[h] = 1.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) sacc[nt][2 * h] = sacc[nt][2 * h + 1] = 0.f;
      } else {
        alpha[h] = exp2f(m_run[h] - mn);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pv = exp2f(sacc[nt][2 * h + e] - mn);
            sacc[nt][2 * h + e] = pv;
            sum += pv;
          }
      }
      m_run[h] = mn;
      l_run[h] = l_run[h] * alpha[h] + sum;
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i) { O[i][0] *= alpha[0]; O[i][1] *= alpha[0]; O[i][2] *= alpha[1]; O[i][3] *= alpha[1]; }
#pragma unroll
    for (int i = 0; i < NLR; ++i) { Olr[i][0] *= alpha[0]; Olr[i][1] *= alpha[0]; Olr[i][2] *= alpha[1]; Olr[i][3] *= alpha[1]; }

    // ---- O += P V_base, O_lr += P L_V (one 16-key block per k-step)
#pragma unroll
    for (int kk = 0; kk < kNW; ++kk) {
      if (!((mask >> kk) & 1)) continue;
      uint32_t pa[4];
      pa[0] = pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
      pa[1] = pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
      pa[2] = pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
      pa[3] = pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
      const uint32_t vt = st + kNW * L.kv_tile + kk * L.kv_tile;
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        const int mi = lane >> 3;
        const int tok = (lane & 7) + (mi & 1) * 8;
        const int dim = 16 * np + (mi >> 1) * 8;
        uint32_t bb[4];
        ldsm_x4_t(bb, vt + (dim / 64) * 2048 + swz<128>(tok, (dim % 64) * 2));
        mma16816(O[2 * np], pa, bb[0], bb[1]);
        mma16816(O[2 * np + 1], pa, bb[2], bb[3]);
      }
      if (use_lr) {
        const uint32_t lvt = st + 2 * kNW * L.kv_tile + kNW * L.lr_tile + kk * L.lr_tile;
        if constexpr (R >= 16) {
#pragma unroll
          for (int np = 0; np < R / 16; ++np) {
            const int mi = lane >> 3;
            const int tok = (lane & 7) + (mi & 1) * 8;
            const int col = 16 * np + (mi >> 1) * 8;
            uint32_t bb[4];
            ldsm_x4_t(bb, lvt + swz<LR_RB>(tok, col * 2));
            mma16816(Olr[2 * np], pa, bb[0], bb[1]);
            mma16816(Olr[2 * np + 1], pa, bb[2], bb[3]);
          }
        } else {
          uint32_t bb[2];
          ldsm_x2_t(bb, lvt + swz<LR_RB>((lane & 7) + ((lane >> 3) & 1) * 8, 0));
          mma16816(Olr[0], pa, bb[0], bb[1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * stage);
    if (++stage == p.nstage) {
      stage = 0;
      phase ^= 1;
    }
  }

  // ---- epilogue: out = (O + O_lr B_V) / l
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = l_run[h];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    l_run[h] = l;
  }
  float* olr = reinterpret_cast<float*>(smem + L.off_olr);
  const float* bv = reinterpret_cast<const float*>(smem + L.off_bv);
  if (use_lr) {
#pragma unroll
    for (int nt = 0; nt < NLR; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = 16 * warp + g8 + 8 * h;
        olr[r * (R + 4) + 8 * nt + 2 * c4] = Olr[nt][2 * h];
        olr[r * (R + 4) + 8 * nt + 2 * c4 + 1] = Olr[nt][2 * h + 1];
      }
    __syncwarp();
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (!rvalid[h]) continue;
    const int rl = 16 * warp + g8 + 8 * h;
    const int r = row0 + rl;
    const int k = r / g;
    const float inv = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
    __nv_bfloat16* orow = p.out + (static_cast<int64_t>(qs + k) * p.Hq + head * g + r % g) * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int j = 8 * nt + 2 * c4;
      float v0 = O[nt][2 * h], v1 = O[nt][2 * h + 1];
      if (use_lr) {
#pragma unroll 8
        for (int kr = 0; kr < R; ++kr) {
          const float ol = olr[rl * (R + 4) + kr];
          v0 = fmaf(ol, bv[kr * D + j], v0);
          v1 = fmaf(ol, bv[kr * D + j + 1], v1);
        }
      }
      *reinterpret_cast<uint32_t*>(orow + j) = pack_bf16(v0 * inv, v1 * inv);
    }
  }
}

template <int D, int R>
lrkv_status run(const lrkv_config& cfg, const PrefillArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.total_q == 0) return LRKV_OK;
  PrefillParams p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.q_start = a.q_start;
  p.seq_lens = a.seq_lens;
  p.adapter_ids = a.adapter_ids;
  p.block_tables = a.block_tables;
  p.B_K = static_cast<const __nv_bfloat16*>(a.B_K);
  p.B_V = static_cast<const __nv_bfloat16*>(a.B_V);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.status = a.status;
  p.num_blocks = a.num_blocks;
  p.num_seqs = a.num_seqs;
  p.max_blocks = a.max_blocks;
  p.max_seq_len = a.max_seq_len;
  p.n_adapters = a.n_adapters;
  p.Hq = cfg.n_q_heads;
  p.Hkv = cfg.n_kv_heads;
  p.g = cfg.n_q_heads / cfg.n_kv_heads;
  p.has_bk = a.B_K != nullptr;
  p.has_bv = a.B_V != nullptr;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  rope_freqs(cfg, &p.freqs);
  const int stage_bytes = PLayout::make(D, R, 1).stage;
  const int fixed = PLayout::make(D, R, 0).total;
  p.nstage = std::min(4, (kSmemLimit - fixed) / stage_bytes);
  if (p.nstage < 2) return LRKV_ERR_UNSUPPORTED;
  const int smem = PLayout::make(D, R, p.nstage).total;
  CUtensorMap tb, tl;
  if (!make_pool_maps(cfg, a.base_pool, a.lr_pool, a.num_blocks, &tb, &tl)) return LRKV_ERR_CUDA;
  auto kern = prefill_kernel<D, R>;
  static bool attr_set = false;  // idempotent per-process kernel attribute
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) !=
        cudaSuccess)
      return LRKV_ERR_CUDA;
    attr_set = true;
  }
  const int tiles = (a.max_q_len * p.g + BMQ - 1) / BMQ;
  dim3 grid(tiles, cfg.n_kv_heads, a.num_seqs);
  kern<<<grid, kThreads, smem, stream>>>(p, tb, tl);
  return cudaGetLastError() == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

}  // namespace

lrkv_status launch_prefill_bf16(const lrkv_config& cfg, const PrefillArgs& a, cudaStream_t stream) {
  const int D = cfg.head_dim, R = cfg.rank;
#define LRKV_PRE(d, r) \
  if (D == d && R == r) return run<d, r>(cfg, a, stream);
  LRKV_PRE(128, 8) LRKV_PRE(128, 16) LRKV_PRE(128, 32) LRKV_PRE(128, 64)
  LRKV_PRE(64, 8) LRKV_PRE(64, 16) LRKV_PRE(64, 32) LRKV_PRE(64, 64)
#undef LRKV_PRE
  return LRKV_ERR_UNSUPPORTED;
}

}  // namespace lrkv
