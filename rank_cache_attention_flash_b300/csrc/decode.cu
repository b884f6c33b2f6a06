// Decode attention over the paged base + shared-A low-rank cache (bf16).
//
// LRAgent (arXiv 2602.01053), Abstract: one cached context serves every agent;
// each agent's adapter contribution is rebuilt from the low-rank cache at
// attention time, never expanded to full width in memory (Flash-LoRA-
// Attention). Here, per 16-token block and per distinct adapter a of the
// queries reading the block:
//     K_a = K_base + RoPE(L_K B_K,a)          rebuilt in registers, never stored
//     S^T = K_a Q^T * scale                   (tokens x query rows; fp16 operands)
//     online softmax over tokens, per row
//     O   += P V_base,  O_lr += P L_V         (the V term reordered: (P L_V) B_V
//                                              is applied once, after the merge)
// The kernel is persistent: each CTA walks work items (context, query group,
// split of the context's blocks, kv head). One producer warp streams the
// blocks' K/V halves and L_K/L_V tiles with 2-D TMA copies (128-byte swizzle)
// through a ring of mbarrier-guarded stages; four consumer warps take one
// block each per stage with legacy warp MMAs (m16n8k16, fp32 accumulators),
// whose fragments let the rebuilt K stay in registers through RoPE, the base
// add and the score MMA. Each item ends by merging the warps' (m, l, O, O_lr)
// and writing an fp32 partial; lrkv_combine merges the splits and applies B_V.
#include <math_constants.h>

#include <algorithm>

#include "lrkv_device.cuh"
#include "lrkv_internal.h"

namespace lrkv {
namespace {

constexpr int kNW = 4;                    // consumer warps
constexpr int kThreads = (kNW + 1) * 32;  // + one producer warp
constexpr int kMaxRows = 16;              // query rows (queries x heads) per item
constexpr int kMaxSlots = 4;              // distinct adapters per item
constexpr int kSmemLimit = 227 * 1024;

struct DecodeParams {
  const __nv_bfloat16* q;
  const int32_t* ctx_q_start;
  const int32_t* adapter_ids;
  const int32_t* block_tables;
  const int32_t* ctx_lens;
  const __nv_bfloat16* B_K;
  float* part_ml;  // [Nq*Hq][S][2] (m in log2 units, l)
  float* part_o;   // [Nq*Hq][S][D + R]
  int32_t* status;
  int64_t num_blocks;
  int64_t n_items;
  int max_blocks, max_ctx_len, n_adapters, num_ctx, Hq, Hkv, g;
  int qg_size, n_qgroups, n_splits, split_blocks, nstage;
  int has_bk, has_bv;
  float scale_log2;
  RopeFreqs freqs;
};

// Shared-memory layout (byte offsets from a 1024-aligned base).
struct Layout {
  int kv_tile, lr_tile, stage, bk_pitch, bk_slot, d_pitch, acc_pitch;
  int off_bk, off_dtab, off_btab, off_freq, off_acc, off_ml, off_misc, off_bar, total;
  __host__ __device__ static Layout make(int D, int R, int nstage, int slots) {
    Layout L;
    L.kv_tile = 16 * D * 2;
    L.lr_tile = 16 * R * 2;
    L.stage = kNW * (2 * L.kv_tile + 2 * L.lr_tile);
    L.bk_pitch = (D + 8) * 2;        // bytes per B_K row in smem (conflict-free ldmatrix)
    L.bk_slot = R * L.bk_pitch;
    L.d_pitch = (D / 2) * 8 + 64;    // delta-table row: D/2 float2 + pad
    L.acc_pitch = D + R + 4;         // floats
    int o = nstage * L.stage;
    L.off_bk = o;   o += slots * L.bk_slot;
    o = (o + 15) & ~15;
    L.off_dtab = o; o += 16 * L.d_pitch;
    L.off_btab = o; o += kNW * (D / 2) * 8;
    L.off_freq = o; o += 2 * 64 * 4;
    L.off_acc = o;  o += kMaxRows * L.acc_pitch * 4;
    L.off_ml = o;   o += 2 * kNW * kMaxRows * 4 + 2 * kMaxRows * 4;
    L.off_misc = o; o += 64;
    o = (o + 7) & ~7;
    L.off_bar = o;  o += 2 * nstage * 8;
    L.total = o + 1024;  // alignment slack
    return L;
  }
};

struct Item {
  int ctx, qg, split, head;
  int q0, nq;      // first query row and count in this group
  int kbeg, kend;  // block range [kbeg, kend)
  int len;
  bool active;
};

__device__ __forceinline__ Item get_item(const DecodeParams& p, int64_t it) {
  Item I;
  I.head = static_cast<int>(it % p.Hkv);
  int64_t r = it / p.Hkv;
  I.split = static_cast<int>(r % p.n_splits);
  r /= p.n_splits;
  I.qg = static_cast<int>(r % p.n_qgroups);
  I.ctx = static_cast<int>(r / p.n_qgroups);
  const int qs = __ldg(p.ctx_q_start + I.ctx), qe = __ldg(p.ctx_q_start + I.ctx + 1);
  I.q0 = qs + I.qg * p.qg_size;
  I.nq = min(p.qg_size, qe - I.q0);
  I.active = I.nq > 0;
  int len = __ldg(p.ctx_lens + I.ctx);
  if (len < 1 || len > p.max_ctx_len) len = 0;
  I.len = len;
  const int nblk = (len + kBlock - 1) / kBlock;
  I.kbeg = I.split * p.split_blocks;
  I.kend = min(I.kbeg + p.split_blocks, nblk);
  return I;
}

template <int D, int R>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeParams p,
                  const __grid_constant__ CUtensorMap tm_base,
                  const __grid_constant__ CUtensorMap tm_lr) {
  constexpr int HALF = D / 2;
  constexpr int NCH = D / 32;   // dim chunks: each covers 16 dims + their RoPE partners
  constexpr int NKS = D / 16;   // k-slices of the score MMA
  constexpr int NRT = R >= 16 ? R / 16 : 1;  // rank k-steps of the rebuild
  constexpr int NLR = R / 8;    // O_lr n-tiles
  constexpr int LR_RB = R * 2;  // low-rank tile row bytes

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const Layout L = Layout::make(D, R, p.nstage, p.qg_size);
  const uint32_t sbase = smem_u32(smem);
  float2* dtab = reinterpret_cast<float2*>(smem + L.off_dtab);
  float* freq = reinterpret_cast<float*>(smem + L.off_freq);
  float* acc = reinterpret_cast<float*>(smem + L.off_acc);
  float* sm_m = reinterpret_cast<float*>(smem + L.off_ml);
  float* sm_l = sm_m + kNW * kMaxRows;
  float* sm_M = sm_l + kNW * kMaxRows;
  float* sm_L = sm_M + kMaxRows;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.off_misc);
  int* stage_mask = reinterpret_cast<int*>(smem + L.off_misc + 16);  // nstage <= 8
  const uint32_t bar_full = sbase + L.off_bar;
  const uint32_t bar_empty = bar_full + 8 * p.nstage;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, c4 = lane & 3;

  // ---- CTA prologue: frequencies, delta table, barriers
  if (tid < HALF) {
    freq[tid] = p.freqs.hi[tid];
    freq[64 + tid] = p.freqs.lo[tid];
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < p.nstage; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kNW);
    }
    mbar_fence_init();
  }
  __syncthreads();
  for (int i = tid; i < 16 * HALF; i += kThreads) {
    const int dl = i / HALF, j = i % HALF;
    float2 cs = rope_cos_sin(dl, freq[j], freq[64 + j]);
    *reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(dtab) + dl * L.d_pitch + j * 8) = cs;
  }
  __syncthreads();

  // ======================================================== producer warp
  if (warp == kNW) {
    if (lane == 0) {
      prefetch_tmap(&tm_base);
      prefetch_tmap(&tm_lr);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // bit s: stage s ever armed
      bool ok = true;
      for (int64_t it = blockIdx.x; ok && it < p.n_items; it += gridDim.x) {
        const Item I = get_item(p, it);
        if (!I.active) continue;
        for (int kb = I.kbeg; kb < I.kend; kb += kNW) {
          if (*abort_flag || !mbar_wait(bar_empty + 8 * stage, phase ^ 1, p.status)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          int mask = 0;
          int blks[kNW];
          uint32_t bytes = 0;
#pragma unroll
          for (int w = 0; w < kNW; ++w) {
            blks[w] = -1;
            const int b = kb + w;
            if (b >= I.kend) continue;
            const int blk = __ldg(p.block_tables + static_cast<int64_t>(I.ctx) * p.max_blocks + b);
            if (blk < 0 || blk >= p.num_blocks) {
              report(p.status, LRKV_ERR_INDEX);
              continue;
            }
            blks[w] = blk;
            mask |= 1 << w;
            bytes += 2 * L.kv_tile + (p.has_bk ? L.lr_tile : 0) + (p.has_bv ? L.lr_tile : 0);
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
            const int yk = ((blk * 2 + 0) * p.Hkv + I.head) * kBlock;
            const int yv = ((blk * 2 + 1) * p.Hkv + I.head) * kBlock;
            const uint32_t kt = st + w * L.kv_tile;
            const uint32_t vt = st + kNW * L.kv_tile + w * L.kv_tile;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
              tma_load_2d(kt + h * 2048, &tm_base, 64 * h, yk, fb);
              tma_load_2d(vt + h * 2048, &tm_base, 64 * h, yv, fb);
            }
            const uint32_t lk = st + 2 * kNW * L.kv_tile + w * L.lr_tile;
            const uint32_t lv = lk + kNW * L.lr_tile;
            if (p.has_bk) tma_load_2d(lk, &tm_lr, 0, (blk * 2 + 0) * kBlock, fb);
            if (p.has_bv) tma_load_2d(lv, &tm_lr, 0, (blk * 2 + 1) * kBlock, fb);
          }
          if (++stage == p.nstage) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: never leave the CTA with copies in flight (bounded waits).
      if (!ok) {
        for (int s = 0; s < p.nstage; ++s)
          if (issued >> s & 1) {
            const uint32_t par = (s < stage) ? phase : (phase ^ 1);
            mbar_wait(bar_full + 8 * s, par, nullptr, 1u << 16);
          }
      }
    }
    return;
  }

  // ======================================================= consumer warps
  float2* btab = reinterpret_cast<float2*>(smem + L.off_btab) + warp * HALF;
  int stage = 0;
  uint32_t phase = 0;

  for (int64_t it = blockIdx.x; it < p.n_items; it += gridDim.x) {
    const Item I = get_item(p, it);
    if (!I.active) continue;
    const int rows = I.nq * p.g;
    const int RN = rows > 8 ? 2 : 1;

    named_bar_sync(1, kNW * 32);  // previous item's merge finished with smem

    // --- distinct adapters of this query group (warp-uniform)
    int slot_ad[kMaxSlots];
    int nslots = 0;
    int qslot[kMaxSlots];  // slot of query qi (qi < qg_size <= kMaxSlots)
#pragma unroll
    for (int i = 0; i < kMaxSlots; ++i) { slot_ad[i] = -1; qslot[i] = 0; }
#pragma unroll
    for (int qi = 0; qi < kMaxSlots; ++qi) {
      if (qi >= I.nq) break;
      int a = __ldg(p.adapter_ids + I.q0 + qi);
      if (a < -1 || a >= p.n_adapters) a = -1;  // reported by the combine
      if (!p.has_bk) a = -1;
      int s = -1;
#pragma unroll
      for (int k = 0; k < kMaxSlots; ++k)
        if (k < nslots && slot_ad[k] == a) s = k;
      if (s < 0) {
        s = nslots++;
#pragma unroll
        for (int k = 0; k < kMaxSlots; ++k)
          if (k == s) slot_ad[k] = a;
      }
#pragma unroll
      for (int k = 0; k < kMaxSlots; ++k)
        if (k == qi) qslot[k] = s;
    }
    // slot of this lane's score columns (rows rn*8 + 2*c4 + e) and per-slot row-tile mask
    int rslot[2][2];
    int slot_rn[kMaxSlots];
#pragma unroll
    for (int k = 0; k < kMaxSlots; ++k) slot_rn[k] = 0;
#pragma unroll
    for (int rn = 0; rn < 2; ++rn)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int row = rn * 8 + 2 * c4 + e;
        const int qi = row < rows ? row / p.g : 0;
        int s = 0;
#pragma unroll
        for (int k = 0; k < kMaxSlots; ++k)
          if (k == qi) s = qslot[k];
        rslot[rn][e] = s;
      }
    for (int row = 0; row < rows; ++row) {
      const int qi = row / p.g;
      int s = 0;
#pragma unroll
      for (int k = 0; k < kMaxSlots; ++k)
        if (k == qi) s = qslot[k];
#pragma unroll
      for (int k = 0; k < kMaxSlots; ++k)
        if (k == s) slot_rn[k] |= 1 << (row >> 3);
    }

    // --- query fragments (B operand of S^T = K Q^T), straight from global
    uint32_t qf[2][NKS][2];
#pragma unroll
    for (int rn = 0; rn < 2; ++rn) {
      const int row = rn * 8 + g8;
      const bool ok = row < rows;
      const __nv_bfloat16* qrow =
          p.q + (static_cast<int64_t>(I.q0 + (ok ? row / p.g : 0)) * p.Hq + I.head * p.g +
                 (ok ? row % p.g : 0)) * D;
#pragma unroll
      for (int ks = 0; ks < NKS; ++ks) {
        qf[rn][ks][0] = ok ? bf16x2_to_f16x2(__ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c4))) : 0u;
        qf[rn][ks][1] = ok ? bf16x2_to_f16x2(__ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c4 + 8))) : 0u;
      }
    }

    // --- B_K slices of the rebuild slots -> smem [slot][k][D] (padded rows)
    {
      const int ctid = tid;  // 0 .. kNW*32-1
      constexpr int VPR = D / 8;  // 16-byte vectors per row
      for (int s = 0; s < nslots; ++s) {
        if (slot_ad[s] < 0) continue;
        const __nv_bfloat16* src = p.B_K + static_cast<int64_t>(slot_ad[s]) * R * p.Hkv * D +
                                   static_cast<int64_t>(I.head) * D;
        uint8_t* dst = smem + L.off_bk + s * L.bk_slot;
        for (int i = ctid; i < R * VPR; i += kNW * 32) {
          const int k = i / VPR, v = i % VPR;
          const uint4 val = __ldg(reinterpret_cast<const uint4*>(src + static_cast<int64_t>(k) * p.Hkv * D) + v);
          *reinterpret_cast<uint4*>(dst + k * L.bk_pitch + v * 16) = val;
        }
      }
    }
    named_bar_sync(1, kNW * 32);

    bool any_rebuild = false;
#pragma unroll
    for (int k = 0; k < kMaxSlots; ++k)
      if (k < nslots && slot_ad[k] >= 0) any_rebuild = true;

    float O[D / 8][4];
    float Olr[NLR][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
#pragma unroll
    for (int i = 0; i < NLR; ++i) Olr[i][0] = Olr[i][1] = Olr[i][2] = Olr[i][3] = 0.f;
    float m_run[2][2], l_run[2][2];
#pragma unroll
    for (int rn = 0; rn < 2; ++rn)
#pragma unroll
      for (int e = 0; e < 2; ++e) { m_run[rn][e] = -CUDART_INF_F; l_run[rn][e] = 0.f; }

    if (I.len == 0 && c4 == 0 && g8 == 0 && warp == 0) report(p.status, LRKV_ERR_INDEX);

    // ------------------------------------------------------ block sweep
    for (int kb = I.kbeg; kb < I.kend; kb += kNW) {
      bool ok = !(*abort_flag) && mbar_wait(bar_full + 8 * stage, phase, p.status);
      if (!ok) *abort_flag = 1;
      const int mask = ok ? stage_mask[stage] : 0;
      const int b = kb + warp;
      if (b < I.kend && (mask >> warp & 1)) {
        const int t0 = b * kBlock;
        const uint32_t st = sbase + stage * L.stage;
        const uint32_t kt = st + warp * L.kv_tile;
        const uint32_t vt = st + kNW * L.kv_tile + warp * L.kv_tile;
        const uint32_t lkt = st + 2 * kNW * L.kv_tile + warp * L.lr_tile;
        const uint32_t lvt = lkt + kNW * L.lr_tile;

        // Rows past the context end may hold stale pool memory: zero their V and
        // L_V rows so that P = 0 there cannot meet a NaN in the PV products.
        if (t0 + kBlock > I.len) {
          const int r0 = I.len - t0;
          for (int i = lane; i < (kBlock - r0) * (D / 8); i += 32) {
            const int r = r0 + i / (D / 8), v = i % (D / 8);
            const uint32_t a = vt + (v / 8) * 2048 + r * 128 + (v % 8) * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(a), "r"(0u) : "memory");
          }
          for (int i = lane; i < (kBlock - r0) * (R / 8); i += 32) {
            const int r = r0 + i / (R / 8), v = i % (R / 8);
            const uint32_t a = lvt + r * LR_RB + v * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(a), "r"(0u) : "memory");
          }
          asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
          __syncwarp();
        }
        // base rotation of this block: e^{i t0 theta_j}
        if (any_rebuild) {
          for (int j = lane; j < HALF; j += 32) btab[j] = rope_cos_sin(t0, freq[j], freq[64 + j]);
          __syncwarp();
        }
        // L_K A fragments (tokens x rank)
        uint32_t alk[NRT][4];
        if (any_rebuild) {
          if constexpr (R >= 16) {
#pragma unroll
            for (int ks = 0; ks < NRT; ++ks) {
              const int mi = lane >> 3;
              const int tok = (lane & 7) + (mi & 1) * 8;
              const int byte = (2 * ks + (mi >> 1)) * 16;
              ldsm_x4(alk[ks], lkt + swz<LR_RB>(tok, byte));
            }
          } else {
            uint32_t t2[2];
            const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
            ldsm_x2(t2, lkt + swz<LR_RB>(tok, 0));
            alk[0][0] = t2[0];
            alk[0][1] = t2[1];
            alk[0][2] = alk[0][3] = 0u;
          }
        }

        float sacc[kMaxSlots][2][4];
#pragma unroll
        for (int a = 0; a < kMaxSlots; ++a)
#pragma unroll
          for (int rn = 0; rn < 2; ++rn) sacc[a][rn][0] = sacc[a][rn][1] = sacc[a][rn][2] = sacc[a][rn][3] = 0.f;

#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) {
          // K_base at this lane's fragment positions: [n][h][tk] (bf16 pairs)
          uint32_t kbv[2][2][2];
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int tk = 0; tk < 2; ++tk) {
                const int j = 16 * cc + 8 * n + 2 * c4 + h * HALF;
                const uint32_t addr = kt + (j / 64) * 2048 + swz<128>(g8 + 8 * tk, (j % 64) * 2);
                asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(kbv[n][h][tk]) : "r"(addr));
              }
          // rotation factors for (tk, n, e)
          float2 cs[2][2][2];
          if (any_rebuild) {
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
          }
#pragma unroll
          for (int a = 0; a < kMaxSlots; ++a) {
            if (a >= nslots) break;
            uint32_t A_lo[4], A_hi[4];
            if (slot_ad[a] >= 0) {
              float y[4][4];
#pragma unroll
              for (int i = 0; i < 4; ++i) y[i][0] = y[i][1] = y[i][2] = y[i][3] = 0.f;
              const uint32_t bk = sbase + L.off_bk + a * L.bk_slot;
              if constexpr (R >= 16) {
#pragma unroll
                for (int ks = 0; ks < NRT; ++ks) {
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    // n-tiles (2cc, 2cc+1) [+ D/16 for the rotation partners]
                    const int mi = lane >> 3;
                    const int krow = 16 * ks + (lane & 7) + (mi & 1) * 8;
                    const int ncol = 16 * cc + h * HALF + (mi >> 1) * 8;
                    uint32_t bb[4];
                    ldsm_x4_t(bb, bk + krow * L.bk_pitch + ncol * 2);
                    mma16816(y[2 * h + 0], alk[ks], bb[0], bb[1]);
                    mma16816(y[2 * h + 1], alk[ks], bb[2], bb[3]);
                  }
                }
              } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int krow = lane & 7;
                  const int ncol = 16 * cc + h * HALF + ((lane >> 3) & 1) * 8;
                  uint32_t bb[2];
                  ldsm_x2_t(bb, bk + krow * L.bk_pitch + ncol * 2);
                  mma1688(y[2 * h + 0], alk[0][0], alk[0][1], bb[0]);
                  mma1688(y[2 * h + 1], alk[0][0], alk[0][1], bb[1]);
                }
              }
              // rotate the rebuilt pair (j, j + d/2), add K_base, pack bf16
              float klo[2][4], khi[2][4];
#pragma unroll
              for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int tk = i >> 1, e = i & 1;
                  const float x = y[n][i], yy = y[n + 2][i];
                  const float c = cs[tk][n][e].x, s = cs[tk][n][e].y;
                  const float blo = e ? bf16_hi(kbv[n][0][tk]) : bf16_lo(kbv[n][0][tk]);
                  const float bhi = e ? bf16_hi(kbv[n][1][tk]) : bf16_lo(kbv[n][1][tk]);
                  klo[n][i] = fmaf(x, c, fmaf(-yy, s, blo));
                  khi[n][i] = fmaf(yy, c, fmaf(x, s, bhi));
                }
              A_lo[0] = pack_f16(klo[0][0], klo[0][1]);
              A_lo[1] = pack_f16(klo[0][2], klo[0][3]);
              A_lo[2] = pack_f16(klo[1][0], klo[1][1]);
              A_lo[3] = pack_f16(klo[1][2], klo[1][3]);
              A_hi[0] = pack_f16(khi[0][0], khi[0][1]);
              A_hi[1] = pack_f16(khi[0][2], khi[0][3]);
              A_hi[2] = pack_f16(khi[1][0], khi[1][1]);
              A_hi[3] = pack_f16(khi[1][2], khi[1][3]);
            } else {
              A_lo[0] = bf16x2_to_f16x2(kbv[0][0][0]);
              A_lo[1] = bf16x2_to_f16x2(kbv[0][0][1]);
              A_lo[2] = bf16x2_to_f16x2(kbv[1][0][0]);
              A_lo[3] = bf16x2_to_f16x2(kbv[1][0][1]);
              A_hi[0] = bf16x2_to_f16x2(kbv[0][1][0]);
              A_hi[1] = bf16x2_to_f16x2(kbv[0][1][1]);
              A_hi[2] = bf16x2_to_f16x2(kbv[1][1][0]);
              A_hi[3] = bf16x2_to_f16x2(kbv[1][1][1]);
            }
#pragma unroll
            for (int rn = 0; rn < 2; ++rn) {
              if (!(slot_rn[a] >> rn & 1)) continue;
              mma16816_f16(sacc[a][rn], A_lo, qf[rn][cc][0], qf[rn][cc][1]);
              mma16816_f16(sacc[a][rn], A_hi, qf[rn][cc + NCH][0], qf[rn][cc + NCH][1]);
            }
          }
        }

        // ---- pick each score column from its own adapter's accumulator; mask; scale
        float s[2][4];
#pragma unroll
        for (int rn = 0; rn < 2; ++rn)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = i & 1;
            float v = sacc[0][rn][i];
#pragma unroll
            for (int a = 1; a < kMaxSlots; ++a)
              if (rslot[rn][e] == a) v = sacc[a][rn][i];
            const int tok = t0 + g8 + 8 * (i >> 1);
            s[rn][i] = tok < I.len ? v * p.scale_log2 : -CUDART_INF_F;
          }
        // ---- online softmax (per score column = query row)
        float alpha[2][2];
        float pr[2][4];
#pragma unroll
        for (int rn = 0; rn < 2; ++rn)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float mx = fmaxf(s[rn][e], s[rn][e + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m_run[rn][e], mx);
            float al, p0, p1;
            if (mn == -CUDART_INF_F) {
              al = 1.f; p0 = 0.f; p1 = 0.f;
            } else {
              al = exp2f(m_run[rn][e] - mn);
              p0 = exp2f(s[rn][e] - mn);
              p1 = exp2f(s[rn][e + 2] - mn);
            }
            m_run[rn][e] = mn;
            l_run[rn][e] = l_run[rn][e] * al + p0 + p1;
            alpha[rn][e] = al;
            pr[rn][e] = p0;
            pr[rn][e + 2] = p1;
          }
        // ---- rescale accumulators (rows g8 and g8 + 8 in the PV layout)
        {
          const int src = g8 >> 1;
          const float a00 = __shfl_sync(0xffffffffu, alpha[0][0], src);
          const float a01 = __shfl_sync(0xffffffffu, alpha[0][1], src);
          const float a10 = __shfl_sync(0xffffffffu, alpha[1][0], src);
          const float a11 = __shfl_sync(0xffffffffu, alpha[1][1], src);
          const float ar0 = (g8 & 1) ? a01 : a00;
          const float ar1 = (g8 & 1) ? a11 : a10;
#pragma unroll
          for (int i = 0; i < D / 8; ++i) { O[i][0] *= ar0; O[i][1] *= ar0; O[i][2] *= ar1; O[i][3] *= ar1; }
#pragma unroll
          for (int i = 0; i < NLR; ++i) { Olr[i][0] *= ar0; Olr[i][1] *= ar0; Olr[i][2] *= ar1; Olr[i][3] *= ar1; }
        }
        // ---- P (rows x tokens) A fragment via register transposes
        uint32_t pa[4];
        pa[0] = movm_t(pack_bf16(pr[0][0], pr[0][1]));
        pa[2] = movm_t(pack_bf16(pr[0][2], pr[0][3]));
        if (RN > 1) {
          pa[1] = movm_t(pack_bf16(pr[1][0], pr[1][1]));
          pa[3] = movm_t(pack_bf16(pr[1][2], pr[1][3]));
        } else {
          pa[1] = pa[3] = 0u;
        }
        // ---- O += P V_base
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
        // ---- O_lr += P L_V
        if (p.has_bv) {
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
            const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
            uint32_t bb[2];
            ldsm_x2_t(bb, lvt + swz<LR_RB>(tok, 0));
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

    // ------------------------------------------------ merge the four warps
#pragma unroll
    for (int rn = 0; rn < 2; ++rn)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float l = l_run[rn][e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        l_run[rn][e] = l;
      }
    if (g8 == 0) {
#pragma unroll
      for (int rn = 0; rn < 2; ++rn)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = rn * 8 + 2 * c4 + e;
          sm_m[warp * kMaxRows + row] = m_run[rn][e];
          sm_l[warp * kMaxRows + row] = l_run[rn][e];
        }
    }
    named_bar_sync(1, kNW * 32);
    if (tid < kMaxRows) {
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < kNW; ++w) M = fmaxf(M, sm_m[w * kMaxRows + tid]);
      float Ls = 0.f;
      if (M != -CUDART_INF_F) {
#pragma unroll
        for (int w = 0; w < kNW; ++w) Ls += sm_l[w * kMaxRows + tid] * exp2f(sm_m[w * kMaxRows + tid] - M);
      }
      sm_M[tid] = M;
      sm_L[tid] = Ls;
    }
    {
      float f[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = g8 + 8 * h;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kNW; ++w) M = fmaxf(M, sm_m[w * kMaxRows + row]);
        const float mw = sm_m[warp * kMaxRows + row];
        f[h] = (M == -CUDART_INF_F || mw == -CUDART_INF_F) ? 0.f : exp2f(mw - M);
      }
      // fixed-order accumulation (warp 0 writes, warps 1.. add): reproducible bits
      for (int w = 0; w < kNW; ++w) {
        if (warp == w) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h == 1 && RN == 1) break;
            float* arow = acc + (g8 + 8 * h) * L.acc_pitch;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
              float2* d2 = reinterpret_cast<float2*>(arow + 8 * nt + 2 * c4);
              const float2 v = make_float2(f[h] * O[nt][2 * h], f[h] * O[nt][2 * h + 1]);
              if (w == 0) *d2 = v;
              else { float2 o = *d2; o.x += v.x; o.y += v.y; *d2 = o; }
            }
#pragma unroll
            for (int nt = 0; nt < NLR; ++nt) {
              float2* d2 = reinterpret_cast<float2*>(arow + D + 8 * nt + 2 * c4);
              const float2 v = make_float2(f[h] * Olr[nt][2 * h], f[h] * Olr[nt][2 * h + 1]);
              if (w == 0) *d2 = v;
              else { float2 o = *d2; o.x += v.x; o.y += v.y; *d2 = o; }
            }
          }
        }
        named_bar_sync(1, kNW * 32);
      }
    }
    named_bar_sync(1, kNW * 32);
    // ---- write the partial of each query row
    for (int i = tid; i < rows * (D + R); i += kNW * 32) {
      const int row = i / (D + R), col = i % (D + R);
      const int n = I.q0 + row / p.g, m = I.head * p.g + row % p.g;
      const int64_t rec = (static_cast<int64_t>(n) * p.Hq + m) * p.n_splits + I.split;
      p.part_o[rec * (D + R) + col] = acc[row * L.acc_pitch + col];
    }
    if (tid < rows) {
      const int n = I.q0 + tid / p.g, m = I.head * p.g + tid % p.g;
      const int64_t rec = (static_cast<int64_t>(n) * p.Hq + m) * p.n_splits + I.split;
      p.part_ml[rec * 2 + 0] = sm_M[tid];
      p.part_ml[rec * 2 + 1] = sm_L[tid];
    }
  }
}

// ---------------------------------------------------------------- combine
// Merges the splits of each (query, head) with log-sum-exp weights, applies
// the reordered V term O_lr B_V,a once, divides by l and stores bf16.
struct CombineParams {
  const float* part_ml;
  const float* part_o;
  const int32_t* adapter_ids;
  const __nv_bfloat16* B_V;
  __nv_bfloat16* out;
  int32_t* status;
  int num_queries, Hq, Hkv, g, n_splits, n_adapters, has_bv;
};

template <int D, int R>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
  __shared__ float wsm[8][256];
  __shared__ float olr[8][R];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t pair = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (pair >= static_cast<int64_t>(p.num_queries) * p.Hq) return;
  const int n = static_cast<int>(pair / p.Hq), m = static_cast<int>(pair % p.Hq);
  const int S = p.n_splits;
  int a = __ldg(p.adapter_ids + n);
  bool bad = a < -1 || a >= p.n_adapters;
  if (bad && lane == 0 && m == 0) report(p.status, LRKV_ERR_INDEX);
  const float* ml = p.part_ml + pair * S * 2;
  float M = -CUDART_INF_F;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, ml[2 * s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float Ls = 0.f;
  for (int s = lane; s < S; s += 32) {
    const float ms = ml[2 * s];
    const float w = (M == -CUDART_INF_F || ms == -CUDART_INF_F) ? 0.f : exp2f(ms - M);
    wsm[warp][s] = w;
    Ls += w * ml[2 * s + 1];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
  __syncwarp();
  const float* po = p.part_o + pair * S * (D + R);
  const bool use_lr = p.has_bv && a >= 0 && !bad;
  for (int k = lane; k < R; k += 32) {
    float v = 0.f;
    if (use_lr)
      for (int s = 0; s < S; ++s) v += wsm[warp][s] * po[static_cast<int64_t>(s) * (D + R) + D + k];
    olr[warp][k] = v;
  }
  __syncwarp();
  const float inv = (Ls > 0.f && !bad) ? 1.f / Ls : 0.f;
  const int kvh = m / p.g;
  for (int j = lane; j < D; j += 32) {
    float v = 0.f;
    for (int s = 0; s < S; ++s) v += wsm[warp][s] * po[static_cast<int64_t>(s) * (D + R) + j];
    if (use_lr) {
      const __nv_bfloat16* bv = p.B_V + static_cast<int64_t>(a) * R * p.Hkv * D + kvh * D + j;
#pragma unroll 8
      for (int k = 0; k < R; ++k) v += olr[warp][k] * __bfloat162float(bv[static_cast<int64_t>(k) * p.Hkv * D]);
    }
    p.out[pair * D + j] = __float2bfloat16_rn(v * inv);
  }
}

template <int D, int R>
lrkv_status run(const lrkv_config& cfg, const DecodeArgs& a, const DecodePlan& plan,
                void* workspace, cudaStream_t stream) {
  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.ctx_q_start = a.ctx_q_start;
  p.adapter_ids = a.adapter_ids;
  p.block_tables = a.block_tables;
  p.ctx_lens = a.ctx_lens;
  p.B_K = static_cast<const __nv_bfloat16*>(a.B_K);
  const int64_t nrec = static_cast<int64_t>(a.num_queries) * cfg.n_q_heads * plan.n_splits;
  p.part_ml = static_cast<float*>(workspace);
  p.part_o = p.part_ml + ((nrec * 2 + 63) / 64) * 64;
  p.status = a.status;
  p.num_blocks = a.num_blocks;
  p.n_items = plan.n_items;
  p.max_blocks = a.max_blocks;
  p.max_ctx_len = a.max_ctx_len;
  p.n_adapters = a.n_adapters;
  p.num_ctx = a.num_ctx;
  p.Hq = cfg.n_q_heads;
  p.Hkv = cfg.n_kv_heads;
  p.g = plan.g;
  p.qg_size = plan.qg_size;
  p.n_qgroups = plan.n_qgroups;
  p.n_splits = plan.n_splits;
  p.split_blocks = plan.split_blocks;
  p.nstage = plan.nstage;
  p.has_bk = a.B_K != nullptr;
  p.has_bv = a.B_V != nullptr;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  rope_freqs(cfg, &p.freqs);

  CUtensorMap tb, tl;
  if (!make_pool_maps(cfg, a.base_pool, a.lr_pool, a.num_blocks, &tb, &tl)) return LRKV_ERR_CUDA;

  if (plan.n_items > 0) {
    auto kern = decode_kernel<D, R>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem_bytes) !=
        cudaSuccess)
      return LRKV_ERR_CUDA;
    kern<<<plan.grid, kThreads, plan.smem_bytes, stream>>>(p, tb, tl);
    if (cudaGetLastError() != cudaSuccess) return LRKV_ERR_CUDA;
  }
  CombineParams c{};
  c.part_ml = p.part_ml;
  c.part_o = p.part_o;
  c.adapter_ids = a.adapter_ids;
  c.B_V = static_cast<const __nv_bfloat16*>(a.B_V);
  c.out = static_cast<__nv_bfloat16*>(a.out);
  c.status = a.status;
  c.num_queries = a.num_queries;
  c.Hq = cfg.n_q_heads;
  c.Hkv = cfg.n_kv_heads;
  c.g = plan.g;
  c.n_splits = plan.n_splits;
  c.n_adapters = a.n_adapters;
  c.has_bv = a.B_V != nullptr;
  const int64_t pairs = static_cast<int64_t>(a.num_queries) * cfg.n_q_heads;
  if (pairs > 0) {
    combine_kernel<D, R><<<static_cast<unsigned>((pairs + 7) / 8), 256, 0, stream>>>(c);
    if (cudaGetLastError() != cudaSuccess) return LRKV_ERR_CUDA;
  }
  return LRKV_OK;
}

}  // namespace

bool plan_decode_bf16(const lrkv_config& cfg, int num_queries, int num_ctx, int max_ctx_len,
                      int max_q_per_ctx, int sm_count, DecodePlan* plan) {
  const int D = cfg.head_dim, R = cfg.rank;
  DecodePlan P{};
  P.g = cfg.n_q_heads / cfg.n_kv_heads;
  if (P.g < 1 || P.g > kMaxRows) return false;
  int qg = std::min(kMaxRows / P.g, kMaxSlots);
  auto bk_bytes = [&](int slots) { return slots * R * (D + 8) * 2; };
  while (qg > 1 && bk_bytes(qg) > 40 * 1024) --qg;
  P.qg_size = qg;
  const int stage_bytes = Layout::make(D, R, 1, qg).stage;
  const int fixed = Layout::make(D, R, 0, qg).total;
  P.nstage = std::min(4, (kSmemLimit - fixed) / stage_bytes);
  if (P.nstage < 2) return false;
  P.smem_bytes = Layout::make(D, R, P.nstage, qg).total;
  P.n_qgroups = std::max(1, (max_q_per_ctx + qg - 1) / qg);
  const int nblk = std::max(1, (max_ctx_len + kBlock - 1) / kBlock);
  const int64_t pairs = static_cast<int64_t>(num_ctx) * P.n_qgroups * cfg.n_kv_heads;
  int best_s = 1;
  double best_eff = -1.0;
  const int smax = std::min(nblk, 256);
  for (int s = 1; s <= smax; ++s) {
    const int sb = (nblk + s - 1) / s;
    const int ss = (nblk + sb - 1) / sb;
    if (ss != s) continue;
    const int64_t items = pairs * s;
    const int64_t waves = (items + sm_count - 1) / sm_count;
    const double eff = static_cast<double>(items) / static_cast<double>(waves * sm_count);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best_s = s;
    }
    if (eff >= 0.95) break;
  }
  P.split_blocks = (nblk + best_s - 1) / best_s;
  P.n_splits = (nblk + P.split_blocks - 1) / P.split_blocks;
  P.n_items = pairs * P.n_splits;
  P.grid = static_cast<int>(std::min<int64_t>(P.n_items, sm_count));
  const int64_t nrec = static_cast<int64_t>(num_queries) * cfg.n_q_heads * P.n_splits;
  P.ws_bytes = static_cast<size_t>((((nrec * 2 + 63) / 64) * 64 + nrec * (D + R)) * 4);
  *plan = P;
  return true;
}

lrkv_status launch_decode_bf16(const lrkv_config& cfg, const DecodeArgs& a,
                               const DecodePlan& plan, void* workspace, cudaStream_t stream) {
  const int D = cfg.head_dim, R = cfg.rank;
#define LRKV_DEC(d, r) \
  if (D == d && R == r) return run<d, r>(cfg, a, plan, workspace, stream);
  LRKV_DEC(128, 8) LRKV_DEC(128, 16) LRKV_DEC(128, 32) LRKV_DEC(128, 64)
  LRKV_DEC(64, 8) LRKV_DEC(64, 16) LRKV_DEC(64, 32) LRKV_DEC(64, 64)
#undef LRKV_DEC
  return LRKV_ERR_UNSUPPORTED;
}

}  // namespace lrkv
