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
// split of the context's blocks, kv head; kv head fastest so that concurrent
// CTAs share the low-rank tiles through L2). Its eight warps take the item's
// blocks round-robin; each warp streams its own blocks (K/V halves with a
// 128-byte swizzle, L_K / L_V tiles) through a private two-stage ring of 2-D
// TMA copies completed on mbarriers, fetching block ids one step ahead and
// crossing item boundaries without draining. Scores of every adapter
// accumulate into one fragment: the query fragment is masked to that
// adapter's rows. Each item ends by merging the warps' (m, l, O, O_lr) in a
// fixed order and writing an fp32 partial; combine_kernel (launched with
// programmatic dependent launch) merges the splits and applies B_V.
#include <math_constants.h>

#include <algorithm>
#include <climits>

#include "lrkv_device.cuh"
#include "lrkv_internal.h"

namespace lrkv {
namespace {

constexpr int kNW = 8;               // warps per CTA (all consume; lane 0 of each issues its TMA)
constexpr int kThreads = kNW * 32;
constexpr int kNST = 2;              // stages per warp
constexpr int kMaxRows = 16;         // query rows (queries x heads) per item
constexpr int kMaxSlots = 4;         // distinct adapters per item
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
  int qg_size, n_qgroups, n_splits, split_blocks;
  int has_bk, has_bv;
  float scale_log2;
  RopeFreqs freqs;
};

// Shared-memory layout (byte offsets from a 1024-aligned base), fixed per (D, R).
// B_K slots: up to four distinct adapters per item (one at rank 64, where the
// ring of 12 KB blocks leaves room for one 17 KB slice).
template <int D, int R>
struct DL {
  static constexpr int kSlots = R >= 64 ? 1 : kMaxSlots;
  static constexpr int kv_tile = 16 * D * 2;
  static constexpr int lr_tile = 16 * R * 2;
  static constexpr int blk = ((2 * kv_tile + 2 * lr_tile) + 1023) & ~1023;  // K, V, L_K, L_V
  static constexpr int bk_pitch = (D + 8) * 2;  // bytes per B_K row (conflict-free ldmatrix)
  static constexpr int bk_slot = R * bk_pitch;
  static constexpr int d_pitch = (D / 2) * 8 + 64;  // delta-table row: D/2 float2 + pad
  static constexpr int acc_pitch = D + R + 4;       // floats; the merge accumulator aliases B_K
  static constexpr int bk_bytes = kSlots * bk_slot;
  static constexpr int acc_bytes = kMaxRows * acc_pitch * 4;
  static constexpr int off_bk = kNW * kNST * blk;
  static constexpr int off_dtab = (off_bk + (bk_bytes > acc_bytes ? bk_bytes : acc_bytes) + 15) & ~15;
  static constexpr int off_btab = off_dtab + 16 * d_pitch;
  static constexpr int off_freq = off_btab + kNW * (D / 2) * 8;
  static constexpr int off_ml = off_freq + 2 * 64 * 4;
  static constexpr int off_misc = off_ml + 2 * kNW * kMaxRows * 4 + 2 * kMaxRows * 4;
  static constexpr int off_bar = (off_misc + 128 + 7) & ~7;
  static constexpr int total = off_bar + kNW * kNST * 8 + 1024;  // + alignment slack
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

// A warp's walk over its (item, block) pairs: items it = blockIdx.x + k * gridDim.x,
// blocks kbeg + warp, kbeg + warp + kNW, ... of each active item.
struct Walk {
  int64_t it;
  int kb;
  Item I;
  bool more;
};

__device__ __forceinline__ void walk_next(const DecodeParams& p, int warp, Walk& w) {
  w.kb += kNW;
  while (!(w.I.active && w.kb < w.I.kend)) {
    w.it += gridDim.x;
    if (w.it >= p.n_items) {
      w.more = false;
      return;
    }
    w.I = get_item(p, w.it);
    w.kb = w.I.kbeg + warp;
  }
  w.more = true;
}

__device__ __forceinline__ void walk_init(const DecodeParams& p, int warp, Walk& w) {
  w.it = static_cast<int64_t>(blockIdx.x) - gridDim.x;
  w.I.active = false;
  w.I.kend = 0;
  w.kb = 0;
  walk_next(p, warp, w);
}

template <int D, int R, int RN>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeParams p,
                  const __grid_constant__ CUtensorMap tm_base,
                  const __grid_constant__ CUtensorMap tm_lr) {
  constexpr int HALF = D / 2;
  constexpr int NCH = D / 32;   // dim chunks: each covers 16 dims + their RoPE partners
  constexpr int NKS = D / 16;   // k-slices of the score MMA
  constexpr int NRT = R >= 16 ? R / 16 : 1;  // rank k-steps of the rebuild
  constexpr int NMT = D / 16;   // m-tiles of O^T (head dims)
  constexpr int NLM = R >= 16 ? R / 16 : 1;  // m-tiles of O_lr^T (rank)
  constexpr int LR_RB = R * 2;  // low-rank tile row bytes

  // The combine kernel may be scheduled now; it waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  using L = DL<D, R>;
  const uint32_t sbase = smem_u32(smem);
  float2* dtab = reinterpret_cast<float2*>(smem + L::off_dtab);
  float* freq = reinterpret_cast<float*>(smem + L::off_freq);
  float* acc = reinterpret_cast<float*>(smem + L::off_bk);  // merge accumulator (aliases B_K)
  float* sm_m = reinterpret_cast<float*>(smem + L::off_ml);
  float* sm_l = sm_m + kNW * kMaxRows;
  float* sm_M = sm_l + kNW * kMaxRows;
  float* sm_L = sm_M + kMaxRows;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::off_misc);
  int* slot_ad_s = reinterpret_cast<int*>(smem + L::off_misc + 16);  // [kMaxSlots]
  int* slot_rn_s = slot_ad_s + kMaxSlots;                             // [kMaxSlots]
  int* q_ad_s = slot_rn_s + kMaxSlots;                                // [kMaxSlots]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, c4 = lane & 3;
  const uint32_t bar0 = sbase + L::off_bar + warp * kNST * 8;  // this warp's ring barriers
  const uint32_t ring0 = sbase + warp * kNST * L::blk;           // this warp's ring

  // ---- CTA prologue: frequencies, delta table, barriers
  if (tid < HALF) {
    freq[tid] = p.freqs.hi[tid];
    freq[64 + tid] = p.freqs.lo[tid];
  }
  if (tid == 0) *abort_flag = 0;
  if (lane == 0) {
    for (int s = 0; s < kNST; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_fence_init();
  }
  __syncthreads();
  for (int i = tid; i < 16 * HALF; i += kThreads) {
    const int dl = i / HALF, j = i % HALF;
    *reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(dtab) + dl * L::d_pitch + j * 8) =
        rope_cos_sin_fast(dl, freq[j], freq[64 + j]);
  }
  if (lane == 0) {
    prefetch_tmap(&tm_base);
    prefetch_tmap(&tm_lr);
  }
  __syncthreads();

  // ---- this warp's TMA ring: issue walk (lane 0 holds the next block id)
  Walk wi;
  walk_init(p, warp, wi);
  int pend_id = -1;
  if (lane == 0 && wi.more)
    pend_id = __ldg(p.block_tables + static_cast<int64_t>(wi.I.ctx) * p.max_blocks + wi.kb);
  uint32_t issued = 0, consumed = 0;
  uint32_t valid_bits = 0;  // bit s: stage s holds a loaded block
  const uint32_t lr_bytes = (p.has_bk ? L::lr_tile : 0) + (p.has_bv ? L::lr_tile : 0);

  auto issue_one = [&]() {
    if (!wi.more) return;
    const int s = issued % kNST;
    int ok = 0;
    if (lane == 0) {
      const int blk = pend_id;
      if (blk < 0 || blk >= p.num_blocks) {
        report(p.status, LRKV_ERR_INDEX);
        mbar_arrive(bar0 + 8 * s);  // complete this stage's phase without data
      } else {
        ok = 1;
        const uint32_t fb = bar0 + 8 * s;
        mbar_arrive_expect_tx(fb, 2 * L::kv_tile + lr_bytes);
        const uint32_t kt = ring0 + s * L::blk, vt = kt + L::kv_tile;
        const uint32_t lk = kt + 2 * L::kv_tile, lv = lk + L::lr_tile;
        const int yk = ((blk * 2 + 0) * p.Hkv + wi.I.head) * kBlock;
        const int yv = ((blk * 2 + 1) * p.Hkv + wi.I.head) * kBlock;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_2d(kt + h * 2048, &tm_base, 64 * h, yk, fb);
          tma_load_2d(vt + h * 2048, &tm_base, 64 * h, yv, fb);
        }
        if (p.has_bk) tma_load_2d(lk, &tm_lr, 0, (blk * 2 + 0) * kBlock, fb);
        if (p.has_bv) tma_load_2d(lv, &tm_lr, 0, (blk * 2 + 1) * kBlock, fb);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    valid_bits = ok ? (valid_bits | (1u << s)) : (valid_bits & ~(1u << s));
    ++issued;
    walk_next(p, warp, wi);
    if (lane == 0 && wi.more)
      pend_id = __ldg(p.block_tables + static_cast<int64_t>(wi.I.ctx) * p.max_blocks + wi.kb);
  };
  for (int s = 0; s < kNST; ++s) issue_one();

  float2* btab = reinterpret_cast<float2*>(smem + L::off_btab) + warp * HALF;

  for (int64_t it = blockIdx.x; it < p.n_items; it += gridDim.x) {
    const Item I = get_item(p, it);
    if (!I.active) continue;
    const int rows = I.nq * p.g;  // <= 8 * RN by the plan

    __syncthreads();  // previous item's merge finished with the B_K / acc / slot smem
    // --- adapter ids of the group's queries (one load per query, in parallel)
    if (tid < I.nq) {
      int a = __ldg(p.adapter_ids + I.q0 + tid);
      if (a < -1 || a >= p.n_adapters || !p.has_bk) a = -1;  // bad ids: reported by the combine
      q_ad_s[tid] = a;
    }
    __syncthreads();
    // distinct adapters (slots), computed redundantly by every thread
    int nslots = 0, qslot[kMaxSlots], sad[kMaxSlots], srn[kMaxSlots];
#pragma unroll
    for (int k = 0; k < kMaxSlots; ++k) { qslot[k] = 0; sad[k] = -2; srn[k] = 0; }
#pragma unroll
    for (int qi = 0; qi < kMaxSlots; ++qi) {
      if (qi < I.nq) {
        const int a = q_ad_s[qi];
        int sl = nslots;
#pragma unroll
        for (int k = 0; k < kMaxSlots; ++k)
          if (k < nslots && sad[k] == a) sl = k;
        if (sl == nslots) {
#pragma unroll
          for (int k = 0; k < kMaxSlots; ++k)
            if (k == sl) sad[k] = a;
          ++nslots;
        }
        int m = 0;
        for (int gi = 0; gi < p.g; ++gi) m |= 1 << ((qi * p.g + gi) >> 3);
#pragma unroll
        for (int k = 0; k < kMaxSlots; ++k) {
          if (k == sl) srn[k] |= m;
          if (k == qi) qslot[k] = sl;
        }
      }
    }
    bool any_rebuild = false;
#pragma unroll
    for (int k = 0; k < kMaxSlots; ++k) any_rebuild |= sad[k] >= 0;
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < kMaxSlots; ++k) {
        slot_ad_s[k] = sad[k];
        slot_rn_s[k] = srn[k];
      }
    }
    // slot of the query row held by this lane in the score B fragment: row rn*8 + g8
    int myslot[RN];
#pragma unroll
    for (int rn = 0; rn < RN; ++rn) {
      const int row = rn * 8 + g8;
      int sl = -1;
#pragma unroll
      for (int k = 0; k < kMaxSlots; ++k)
        if (row < rows && k == row / p.g) sl = qslot[k];
      myslot[rn] = sl;
    }

    // --- query fragments (B operand of S^T = K Q^T), fp16, straight from global
    uint32_t qf[RN][NKS][2];
#pragma unroll
    for (int rn = 0; rn < RN; ++rn) {
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
    // --- B_K slices of the rebuild slots -> smem [slot][k][D] (padded rows), async copies
    {
      constexpr int VPR = D / 8;  // 16-byte vectors per row
#pragma unroll
      for (int s = 0; s < L::kSlots; ++s) {
        const int a = sad[s];
        if (a < 0) continue;
        const __nv_bfloat16* src = p.B_K + static_cast<int64_t>(a) * R * p.Hkv * D +
                                   static_cast<int64_t>(I.head) * D;
        const uint32_t dst = sbase + L::off_bk + s * L::bk_slot;
        for (int i = tid; i < R * VPR; i += kThreads) {
          const int k = i / VPR, v = i % VPR;
          const void* g = reinterpret_cast<const uint4*>(src + static_cast<int64_t>(k) * p.Hkv * D) + v;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst + k * L::bk_pitch + v * 16),
                       "l"(g) : "memory");
        }
      }
      asm volatile("cp.async.commit_group;\n" ::: "memory");
      asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    }
    __syncthreads();

    // O^T [head dims x query rows] and O_lr^T [rank x query rows] accumulators
    float OT[NMT][RN][4];
    float OlrT[NLM][RN][4];
#pragma unroll
    for (int i = 0; i < NMT; ++i)
#pragma unroll
      for (int rn = 0; rn < RN; ++rn) OT[i][rn][0] = OT[i][rn][1] = OT[i][rn][2] = OT[i][rn][3] = 0.f;
#pragma unroll
    for (int i = 0; i < NLM; ++i)
#pragma unroll
      for (int rn = 0; rn < RN; ++rn) OlrT[i][rn][0] = OlrT[i][rn][1] = OlrT[i][rn][2] = OlrT[i][rn][3] = 0.f;
    float m_run[RN][2], l_run[RN][2];
#pragma unroll
    for (int rn = 0; rn < RN; ++rn)
#pragma unroll
      for (int e = 0; e < 2; ++e) { m_run[rn][e] = -CUDART_INF_F; l_run[rn][e] = 0.f; }

    if (I.len == 0 && tid == 0) report(p.status, LRKV_ERR_INDEX);

    // ------------------------------------------------------ block sweep
    for (int b = I.kbeg + warp; b < I.kend; b += kNW) {
      const int s = consumed % kNST;
      const uint32_t par = (consumed / kNST) & 1;
      const bool have = (valid_bits >> s) & 1;
      // every wait result below is made warp-uniform before any warp-collective use
      bool ok = have && !__shfl_sync(0xffffffffu, *abort_flag, 0);
      if (ok) ok = mbar_wait(bar0 + 8 * s, par, p.status);
      ok = have && __all_sync(0xffffffffu, ok);
      if (have && !ok) *abort_flag = 1;
      if (ok) {
        const int t0 = b * kBlock;
        const uint32_t kt = ring0 + s * L::blk, vt = kt + L::kv_tile;
        const uint32_t lkt = kt + 2 * L::kv_tile, lvt = lkt + L::lr_tile;

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
          __syncwarp();
        }
        // base rotation of this block: e^{i t0 theta_j}
        if (any_rebuild) {
          for (int j = lane; j < HALF; j += 32) btab[j] = rope_cos_sin_fast(t0, freq[j], freq[64 + j]);
          __syncwarp();
        }
        // L_K A fragments (tokens x rank)
        uint32_t alk[NRT][4];
        if (any_rebuild) {
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

        // two independent score accumulators (low / high head-dim halves) keep the
        // MMA dependency chain short
        float sacc[2][RN][4];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int rn = 0; rn < RN; ++rn)
            sacc[hh][rn][0] = sacc[hh][rn][1] = sacc[hh][rn][2] = sacc[hh][rn][3] = 0.f;

#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) {
          // K_base at this lane's fragment positions, as fp16 pairs: [n][h][tk]
          uint32_t kb16[2][2][2];
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int tk = 0; tk < 2; ++tk) {
                const int j = 16 * cc + 8 * n + 2 * c4 + h * HALF;
                const uint32_t addr = kt + (j / 64) * 2048 + swz<128>(g8 + 8 * tk, (j % 64) * 2);
                uint32_t v;
                asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
                kb16[n][h][tk] = bf16x2_to_f16x2(v);
              }
          // rotation factors of this lane's (token, pair) positions as fp16 pairs
          uint32_t c16[2][2], s16[2][2], ns16[2][2];  // [tk][n]
          if (any_rebuild) {
#pragma unroll
            for (int n = 0; n < 2; ++n) {
              const int j = 16 * cc + 8 * n + 2 * c4;
              const float4 bq = *reinterpret_cast<const float4*>(btab + j);
#pragma unroll
              for (int tk = 0; tk < 2; ++tk) {
                const float4 dq = *reinterpret_cast<const float4*>(
                    reinterpret_cast<const uint8_t*>(dtab) + (g8 + 8 * tk) * L::d_pitch + j * 8);
                const float c0 = bq.x * dq.x - bq.y * dq.y, s0 = bq.y * dq.x + bq.x * dq.y;
                const float c1 = bq.z * dq.z - bq.w * dq.w, s1 = bq.w * dq.z + bq.z * dq.w;
                c16[tk][n] = pack_f16(c0, c1);
                s16[tk][n] = pack_f16(s0, s1);
                ns16[tk][n] = pack_f16(-s0, -s1);
              }
            }
          }
#pragma unroll 1
          for (int a = 0; a < nslots; ++a) {
            const int ad = slot_ad_s[a];
            const int rnm = slot_rn_s[a];
            uint32_t A_lo[4], A_hi[4];
            if (ad >= 0) {
              float y[4][4];
#pragma unroll
              for (int i = 0; i < 4; ++i) y[i][0] = y[i][1] = y[i][2] = y[i][3] = 0.f;
              const uint32_t bk = sbase + L::off_bk + a * L::bk_slot;
              if constexpr (R >= 16) {
#pragma unroll
                for (int ks = 0; ks < NRT; ++ks)
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    // n-tiles (2cc, 2cc+1) [+ D/16 for the rotation partners]
                    const int mi = lane >> 3;
                    const int krow = 16 * ks + (lane & 7) + (mi & 1) * 8;
                    const int ncol = 16 * cc + h * HALF + (mi >> 1) * 8;
                    uint32_t bb[4];
                    ldsm_x4_t(bb, bk + krow * L::bk_pitch + ncol * 2);
                    mma16816(y[2 * h + 0], alk[ks], bb[0], bb[1]);
                    mma16816(y[2 * h + 1], alk[ks], bb[2], bb[3]);
                  }
              } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int ncol = 16 * cc + h * HALF + ((lane >> 3) & 1) * 8;
                  uint32_t bb[2];
                  ldsm_x2_t(bb, bk + (lane & 7) * L::bk_pitch + ncol * 2);
                  mma1688(y[2 * h + 0], alk[0][0], alk[0][1], bb[0]);
                  mma1688(y[2 * h + 1], alk[0][0], alk[0][1], bb[1]);
                }
              }
              // rotate the rebuilt pair (j, j + d/2) and add K_base, in packed fp16:
              //   k_lo = K_lo + x cos - y sin,   k_hi = K_hi + y cos + x sin
#pragma unroll
              for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int tk = 0; tk < 2; ++tk) {
                  const uint32_t x = pack_f16(y[n][2 * tk], y[n][2 * tk + 1]);
                  const uint32_t yy = pack_f16(y[n + 2][2 * tk], y[n + 2][2 * tk + 1]);
                  A_lo[2 * n + tk] = hfma2_u32(x, c16[tk][n], hfma2_u32(yy, ns16[tk][n], kb16[n][0][tk]));
                  A_hi[2 * n + tk] = hfma2_u32(yy, c16[tk][n], hfma2_u32(x, s16[tk][n], kb16[n][1][tk]));
                }
            } else {
#pragma unroll
              for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int tk = 0; tk < 2; ++tk) {
                  A_lo[2 * n + tk] = kb16[n][0][tk];
                  A_hi[2 * n + tk] = kb16[n][1][tk];
                }
            }
            // scores of this adapter's rows only: its query fragment, other rows zeroed
#pragma unroll
            for (int rn = 0; rn < RN; ++rn) {
              if (!((rnm >> rn) & 1)) continue;
              const bool mine = myslot[rn] == a;
              const uint32_t q0 = mine ? qf[rn][cc][0] : 0u, q1 = mine ? qf[rn][cc][1] : 0u;
              const uint32_t q2 = mine ? qf[rn][cc + NCH][0] : 0u, q3 = mine ? qf[rn][cc + NCH][1] : 0u;
              mma16816_f16(sacc[0][rn], A_lo, q0, q1);
              mma16816_f16(sacc[1][rn], A_hi, q2, q3);
            }
          }
        }

        // ---- mask and scale (S^T: tokens g8, g8 + 8 x query rows rn*8 + 2*c4 + e)
        float sv[RN][4];
#pragma unroll
        for (int rn = 0; rn < RN; ++rn)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tok = t0 + g8 + 8 * (i >> 1);
            sv[rn][i] = tok < I.len ? (sacc[0][rn][i] + sacc[1][rn][i]) * p.scale_log2 : -CUDART_INF_F;
          }
        // ---- online softmax (per score column = query row)
        float alpha[RN][2];
        float pr[RN][4];
        bool moved = false;
#pragma unroll
        for (int rn = 0; rn < RN; ++rn)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float mx = fmaxf(sv[rn][e], sv[rn][e + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m_run[rn][e], mx);
            float al, p0, p1;
            if (mn == -CUDART_INF_F) {
              al = 1.f; p0 = 0.f; p1 = 0.f;
            } else {
              al = exp2f(m_run[rn][e] - mn);
              p0 = exp2f(sv[rn][e] - mn);
              p1 = exp2f(sv[rn][e + 2] - mn);
            }
            moved |= al != 1.f;
            m_run[rn][e] = mn;
            l_run[rn][e] = l_run[rn][e] * al + p0 + p1;
            alpha[rn][e] = al;
            pr[rn][e] = p0;
            pr[rn][e + 2] = p1;
          }
        // ---- rescale accumulators: this lane's O^T columns are its own score rows
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
          for (int rn = 0; rn < RN; ++rn) {
#pragma unroll
            for (int i = 0; i < NMT; ++i) {
              OT[i][rn][0] *= alpha[rn][0]; OT[i][rn][1] *= alpha[rn][1];
              OT[i][rn][2] *= alpha[rn][0]; OT[i][rn][3] *= alpha[rn][1];
            }
#pragma unroll
            for (int i = 0; i < NLM; ++i) {
              OlrT[i][rn][0] *= alpha[rn][0]; OlrT[i][rn][1] *= alpha[rn][1];
              OlrT[i][rn][2] *= alpha[rn][0]; OlrT[i][rn][3] *= alpha[rn][1];
            }
          }
        }
        // ---- P^T (tokens x rows) B fragments via register transposes
        uint32_t pb[RN][2];
#pragma unroll
        for (int rn = 0; rn < RN; ++rn) {
          pb[rn][0] = movm_t(pack_bf16(pr[rn][0], pr[rn][1]));
          pb[rn][1] = movm_t(pack_bf16(pr[rn][2], pr[rn][3]));
        }
        // ---- O^T += V_base^T P^T (M = head dims, N = query rows, K = tokens)
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
          const int mi = lane >> 3;
          const int tok = (lane & 7) + (mi >> 1) * 8;
          const int dim = 16 * mt + (mi & 1) * 8;
          uint32_t av[4];
          ldsm_x4_t(av, vt + (dim / 64) * 2048 + swz<128>(tok, (dim % 64) * 2));
#pragma unroll
          for (int rn = 0; rn < RN; ++rn) mma16816(OT[mt][rn], av, pb[rn][0], pb[rn][1]);
        }
        // ---- O_lr^T += L_V^T P^T
        if (p.has_bv) {
          if constexpr (R >= 16) {
#pragma unroll
            for (int mt = 0; mt < NLM; ++mt) {
              const int mi = lane >> 3;
              const int tok = (lane & 7) + (mi >> 1) * 8;
              const int col = 16 * mt + (mi & 1) * 8;
              uint32_t av[4];
              ldsm_x4_t(av, lvt + swz<LR_RB>(tok, col * 2));
#pragma unroll
              for (int rn = 0; rn < RN; ++rn) mma16816(OlrT[mt][rn], av, pb[rn][0], pb[rn][1]);
            }
          } else {
            uint32_t t2[2];
            ldsm_x2_t(t2, lvt + swz<LR_RB>((lane & 7) + ((lane >> 3) & 1) * 8, 0));
            const uint32_t av[4] = {t2[0], 0u, t2[1], 0u};  // rank rows 8..15 do not exist
#pragma unroll
            for (int rn = 0; rn < RN; ++rn) mma16816(OlrT[0][rn], av, pb[rn][0], pb[rn][1]);
          }
        }
      }
      // release the stage and refill it with this warp's next block
      ++consumed;
      __syncwarp();
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      if (!__shfl_sync(0xffffffffu, *abort_flag, 0)) issue_one();
    }

    // ------------------------------------------------ merge the warps
#pragma unroll
    for (int rn = 0; rn < RN; ++rn)
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
      for (int rn = 0; rn < RN; ++rn)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = rn * 8 + 2 * c4 + e;
          sm_m[warp * kMaxRows + row] = m_run[rn][e];
          sm_l[warp * kMaxRows + row] = l_run[rn][e];
        }
    }
    __syncthreads();  // also: every warp is past its B_K reads; acc may alias them now
    if (tid < RN * 8) {
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
      // per-row weight of this warp's partial: exp2(m_w - max over warps)
      float f[RN][2];
#pragma unroll
      for (int rn = 0; rn < RN; ++rn)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = rn * 8 + 2 * c4 + e;
          float M = -CUDART_INF_F;
#pragma unroll
          for (int w = 0; w < kNW; ++w) M = fmaxf(M, sm_m[w * kMaxRows + row]);
          const float mw = m_run[rn][e];
          f[rn][e] = (M == -CUDART_INF_F || mw == -CUDART_INF_F) ? 0.f : exp2f(mw - M);
        }
      // fixed-order accumulation (warp 0 writes, warps 1.. add): reproducible bits.
      // acc[row][col]: col = head dim 16*mt + g8 (+8), or D + rank index.
      for (int w = 0; w < kNW; ++w) {
        if (warp == w) {
          float cur[NMT + NLM][RN][4];
          if (w > 0) {  // all loads first, then all stores
#pragma unroll
            for (int i = 0; i < NMT + NLM; ++i)
#pragma unroll
              for (int rn = 0; rn < RN; ++rn)
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  const int row = rn * 8 + 2 * c4 + (v & 1);
                  const int col = (i < NMT ? 16 * i : D + 16 * (i - NMT)) + g8 + 8 * (v >> 1);
                  cur[i][rn][v] = (i >= NMT && 16 * (i - NMT) + g8 + 8 * (v >> 1) >= R)
                                      ? 0.f : acc[row * L::acc_pitch + col];
                }
          }
#pragma unroll
          for (int i = 0; i < NMT + NLM; ++i)
#pragma unroll
            for (int rn = 0; rn < RN; ++rn)
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const int row = rn * 8 + 2 * c4 + (v & 1);
                const int k = (i < NMT ? 16 * i : 16 * (i - NMT)) + g8 + 8 * (v >> 1);
                if (i >= NMT && k >= R) continue;
                const int col = (i < NMT ? 0 : D) + k;
                const float x = f[rn][v & 1] * (i < NMT ? OT[i][rn][v] : OlrT[i - NMT][rn][v]);
                acc[row * L::acc_pitch + col] = (w > 0 ? cur[i][rn][v] : 0.f) + x;
              }
        }
        __syncthreads();
      }
    }
    // ---- write the partial of each query row
    for (int i = tid; i < rows * (D + R); i += kThreads) {
      const int row = i / (D + R), col = i % (D + R);
      const int n = I.q0 + row / p.g, m = I.head * p.g + row % p.g;
      const int64_t rec = (static_cast<int64_t>(n) * p.Hq + m) * p.n_splits + I.split;
      p.part_o[rec * (D + R) + col] = acc[row * L::acc_pitch + col];
    }
    if (tid < rows) {
      const int n = I.q0 + tid / p.g, m = I.head * p.g + tid % p.g;
      const int64_t rec = (static_cast<int64_t>(n) * p.Hq + m) * p.n_splits + I.split;
      p.part_ml[rec * 2 + 0] = sm_M[tid];
      p.part_ml[rec * 2 + 1] = sm_L[tid];
    }
  }
  // Drain: never leave the CTA with copies in flight (bounded waits; only after an abort).
  if (__shfl_sync(0xffffffffu, *abort_flag, 0)) {
    for (uint32_t k = consumed; k < issued; ++k) {
      const int s = k % kNST;
      if ((valid_bits >> s) & 1) mbar_wait(bar0 + 8 * s, (k / kNST) & 1, nullptr, 1u << 16);
    }
  }
}

// ---------------------------------------------------------------- combine
// Merges the splits of each (query, head) with log-sum-exp weights, applies
// the reordered V term O_lr B_V,a once, divides by l and stores bf16.
// One CTA per (query, head); thread t owns column t of the partial rows.
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
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineParams p) {
  constexpr int NCOL = D + R;
  __shared__ float w_s[256];
  __shared__ float red[8];
  __shared__ float olr[R];
  // wait until the decode grid has finished and its partials are visible
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int64_t pair = blockIdx.x;
  const int n = static_cast<int>(pair / p.Hq), m = static_cast<int>(pair % p.Hq);
  const int S = p.n_splits;
  const int a = __ldg(p.adapter_ids + n);
  const bool bad = a < -1 || a >= p.n_adapters;
  if (bad && tid == 0 && m == 0) report(p.status, LRKV_ERR_INDEX);
  const float* ml = p.part_ml + pair * S * 2;
  // max over splits
  float M = -CUDART_INF_F;
  for (int s = tid; s < S; s += 256) M = fmaxf(M, __ldg(ml + 2 * s));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) red[wid] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  float Ls = 0.f;
  for (int s = tid; s < S; s += 256) {
    const float ms = __ldg(ml + 2 * s);
    const float w = (M == -CUDART_INF_F || ms == -CUDART_INF_F) ? 0.f : exp2f(ms - M);
    w_s[s] = w;
    Ls += w * __ldg(ml + 2 * s + 1);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
  if (lane == 0) red[wid] = Ls;
  __syncthreads();
  Ls = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) Ls += red[w];
  const bool use_lr = p.has_bv && a >= 0 && !bad;
  float v = 0.f;
  if (tid < NCOL) {
    const float* po = p.part_o + pair * S * NCOL + tid;
#pragma unroll 8
    for (int s = 0; s < S; ++s) v += w_s[s] * __ldg(po + static_cast<int64_t>(s) * NCOL);
    if (tid >= D) olr[tid - D] = use_lr ? v : 0.f;
  }
  __syncthreads();
  if (tid < D) {
    if (use_lr) {
      const __nv_bfloat16* bv = p.B_V + static_cast<int64_t>(a) * R * p.Hkv * D + (m / p.g) * D + tid;
#pragma unroll 8
      for (int k = 0; k < R; ++k) v = fmaf(olr[k], __bfloat162float(bv[static_cast<int64_t>(k) * p.Hkv * D]), v);
    }
    const float inv = (Ls > 0.f && !bad) ? 1.f / Ls : 0.f;
    p.out[pair * D + tid] = __float2bfloat16_rn(v * inv);
  }
}

template <int D, int R, int RN>
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
  p.has_bk = a.B_K != nullptr;
  p.has_bv = a.B_V != nullptr;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  rope_freqs(cfg, &p.freqs);

  CUtensorMap tb, tl;
  if (!make_pool_maps(cfg, a.base_pool, a.lr_pool, a.num_blocks, &tb, &tl)) return LRKV_ERR_CUDA;

  if (plan.n_items > 0) {
    auto kern = decode_kernel<D, R, RN>;
    static bool attr_set = false;  // idempotent per-process kernel attribute
    if (!attr_set) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) !=
          cudaSuccess)
        return LRKV_ERR_CUDA;
      attr_set = true;
    }
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
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(pairs));
    lc.blockDim = dim3(256);
    lc.dynamicSmemBytes = 0;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (cudaLaunchKernelEx(&lc, combine_kernel<D, R>, c) != cudaSuccess) return LRKV_ERR_CUDA;
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
  int slots = 0, total = 0;
#define LRKV_L(d, r) \
  if (D == d && R == r) { slots = DL<d, r>::kSlots; total = DL<d, r>::total; }
  LRKV_L(128, 8) LRKV_L(128, 16) LRKV_L(128, 32) LRKV_L(128, 64)
  LRKV_L(64, 8) LRKV_L(64, 16) LRKV_L(64, 32) LRKV_L(64, 64)
#undef LRKV_L
  if (slots == 0 || total > kSmemLimit) return false;
  const int qg = std::min(kMaxRows / P.g, slots);
  P.qg_size = qg;
  P.rn = qg * P.g > 8 ? 2 : 1;
  P.nstage = kNST;
  P.smem_bytes = total;
  P.n_qgroups = std::max(1, (max_q_per_ctx + qg - 1) / qg);
  const int nblk = std::max(1, (max_ctx_len + kBlock - 1) / kBlock);
  const int64_t pairs = static_cast<int64_t>(num_ctx) * P.n_qgroups * cfg.n_kv_heads;
  // Splits: as many as keep every SM busy in whole waves of items (>= 0.95
  // efficiency), counting how evenly a split's blocks fall on the kNW warps.
  int best_s = 1;
  double best_eff = -1.0;
  const int smax = std::min(nblk, 256);
  for (int s = 1; s <= smax; ++s) {
    const int sb = (nblk + s - 1) / s;
    const int ss = (nblk + sb - 1) / sb;
    if (ss != s) continue;
    const int64_t items = pairs * s;
    const int64_t waves = (items + sm_count - 1) / sm_count;
    const double rounds = static_cast<double>((sb + kNW - 1) / kNW) * kNW / sb;  // warp balance
    const double eff = static_cast<double>(items) / static_cast<double>(waves * sm_count) / rounds;
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
#define LRKV_DEC(d, r)                                                          \
  if (D == d && R == r)                                                         \
    return plan.rn == 1 ? run<d, r, 1>(cfg, a, plan, workspace, stream)         \
                        : run<d, r, 2>(cfg, a, plan, workspace, stream);
  LRKV_DEC(128, 8) LRKV_DEC(128, 16) LRKV_DEC(128, 32) LRKV_DEC(128, 64)
  LRKV_DEC(64, 8) LRKV_DEC(64, 16) LRKV_DEC(64, 32) LRKV_DEC(64, 64)
#undef LRKV_DEC
  return LRKV_ERR_UNSUPPORTED;
}

}  // namespace lrkv
