// Causal prefill attention over the paged base + shared-A low-rank cache (bf16),
// on the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// LRAgent (arXiv 2602.01053), Abstract (Flash-LoRA-Attention): each agent's
// K adapter term L_K B_K is rebuilt per key tile on chip, rotated and added to
// K_base; the V term is reordered as (P L_V) B_V. PReCache, Abstract: a new
// turn attends over the context cached by earlier agents plus its own chunk.
//
// One CTA per (sequence, kv head, tile of 128 query rows); rows are
// (query, head-in-group) pairs so that the g query heads sharing a kv head
// share every key tile. Per stage of 128 keys (8 paged blocks):
//   Y    = L_K B_K                    tcgen05, 128 keys x d, K = rank  -> TMEM
//   K_a  = K_base + RoPE(Y)           rebuild warpgroup, in place in the
//                                     stage's K tile (fp16, never stored to HBM)
//   S    = Q K_a^T                    tcgen05, Q read from TMEM, two halves of
//                                     64 keys (double-buffered in TMEM)
//   P    = online softmax(S)          softmax warpgroup, thread = query row,
//                                     P written back over S as bf16
//   O   += P V_base, O_lr += P L_V    tcgen05, P read from TMEM
// and at the end out = (O + O_lr B_V) / l.
//
// Warp roles (320 threads): warp 0 streams K, V, L_K, L_V tiles with 2-D TMA
// copies into an mbarrier ring; warp 1 owns the tensor memory and one of its
// lanes issues every MMA (in-order, so a TMEM region is only rewritten after
// the MMAs reading it were issued); warps 2-5 run the softmax; warps 6-9
// rebuild K_a. Tensor-memory columns: Q [0, d/2) packed, S0 [64, 128),
// S1 [128, 192), O [192, 192+d), O_lr [192+d, 192+d+r'), Y [384, 384+d).
// Every wait is bounded: a wait that gives up stores LRKV_ERR_TIMEOUT, sets a
// CTA-wide abort flag, and every role leaves its loop; no MMA or copy is left
// in flight when the tensor memory is released.
#include <math_constants.h>

#include <algorithm>

#include "lrkv_device.cuh"
#include "lrkv_internal.h"
#include "tcgen05.cuh"

namespace lrkv {
namespace {

constexpr int kThreads = 320;
constexpr int BM = 128;   // query rows per CTA (= TMEM lanes)
constexpr int BN = 128;   // keys per stage (8 paged blocks)
constexpr int HN = 64;    // keys per score half-tile
constexpr int kSmemLimit = 227 * 1024;
constexpr uint32_t kTmemCols = 512;
constexpr int Q_COL = 0, S_COL0 = 64, O_COL = 192, Y_COL = 384;
constexpr int kSmWarp0 = 2, kRbWarp0 = 6;  // first softmax / rebuild warp
constexpr float kRescaleLog2 = 8.0f;       // rescale O only when the row max grows by > 2^8

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
  int num_seqs, max_blocks, max_seq_len, n_adapters, Hq, Hkv, g;
  int has_bk, has_bv;
  float scale_log2;
  RopeFreqs freqs;
};

// Y = L_K B_K is produced in column groups of 32: group g holds the 16 dims
// 16g.. and their RoPE partners d/2 + 16g.. (B_K^T is staged with its rows in
// that order), so each group can be rotated on its own and its TMEM columns
// refilled for the next stage as soon as they have been read.
// Shared-memory layout (byte offsets from a 1024-aligned base).
template <int D, int R>
struct PL {
  static constexpr int RP = R < 16 ? 16 : R;      // rank padded to the MMA granularity
  static constexpr int LSPAN = RP * 2;            // bytes per low-rank row (32 / 64 / 128)
  static constexpr int KV = BN * D * 2;           // K or V tile
  static constexpr int LT = BN * LSPAN;           // L_K or L_V tile
  static constexpr int STAGE = 2 * KV + 2 * LT;
  static constexpr int BKB = D * LSPAN;           // B_K^T tile [d][r'], K-major
  static constexpr int BTAB = 8 * (D / 2) * 8;    // per-stage block start angles (cos, sin)
  static constexpr int MISC = 512;
  static constexpr int FIXED = BKB + BTAB + MISC + 1024;
  static constexpr int NST_FIT = (kSmemLimit - FIXED) / STAGE;
  static constexpr int NST = NST_FIT > 4 ? 4 : NST_FIT;
  static constexpr int off_k = 0, off_v = KV, off_lk = 2 * KV, off_lv = 2 * KV + LT;
  static constexpr int off_bk = NST * STAGE;
  static constexpr int off_btab = off_bk + BKB;
  static constexpr int off_misc = off_btab + BTAB;
  static constexpr int total = off_misc + MISC + 1024;  // + alignment slack
  static_assert(NST >= 2, "two pipeline stages must fit");
  static_assert(total <= kSmemLimit, "shared memory");
  static_assert(192 + D + RP <= Y_COL, "tensor-memory columns");
};

// Barrier slots inside the misc area (8 bytes each).
enum : int {
  B_FULL = 0,    // [4] TMA -> consumers (one phase per stage use)
  B_EMPTY = 4,   // [4] MMA commit -> producer
  B_KA = 8,      // [4] rebuild warpgroup -> MMA (K_a written)
  B_YFULL = 12,  // [4] MMA commit -> rebuild (column group of Y in TMEM)
  B_YFREE = 16,  // [4] rebuild -> MMA (column group of Y read)
  B_SFULL = 20,  // [2] MMA commit -> softmax (S half-tile in TMEM)
  B_PFULL = 22,  // [2] softmax -> MMA (P written, O rescaled)
  B_OBAR = 24,   // MMA commit after each P V
  B_DRAIN = 25,  // MMA commit on abort: every issued MMA has completed
  B_EPI = 26,    // softmax -> MMA: fp16(O_lr / l) in TMEM and B_V in smem
  B_ZFULL = 27,  // MMA commit -> softmax: Z = fp16(O_lr / l) B_V in TMEM
  B_COUNT = 28
};

// Non-blocking test of an mbarrier phase (the MMA issuer polls several).
__device__ __forceinline__ bool test_parity(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr long long kWaitCycles = 1ll << 31;  // ~1 s: a wait this long has failed

// 2^x by the hardware approximation (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Waits for an mbarrier phase with try_wait (which suspends until the phase
// completes or a short hardware time limit), without sleeping in between;
// gives up after kWaitCycles, stores LRKV_ERR_TIMEOUT and returns false.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, int32_t* st) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > kWaitCycles) {
      report(st, LRKV_ERR_TIMEOUT);
      return false;
    }
  }
}

// Named barrier over `count` threads that also ORs a predicate across them:
// every participant gets the same answer, so a group can leave a loop together.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

template <int D, int R>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p,
                   const __grid_constant__ CUtensorMap tm_base,
                   const __grid_constant__ CUtensorMap tm_lr) {
  using L = PL<D, R>;
  constexpr int HALF = D / 2;
  constexpr int RP = L::RP;
  constexpr int LSPAN = L::LSPAN;
  constexpr int NST = L::NST;
  constexpr int OLR_COL = O_COL + D;
  constexpr uint32_t SW_LR = tc::swizzle_code(LSPAN);
  constexpr int NG = HALF / 16;  // Y column groups
  constexpr uint32_t kIdY = tc::idesc_f16(128, 32, true, false, false);
  constexpr uint32_t kIdS16 = tc::idesc_f16(128, HN, false, false, false);  // fp16 Q, K_a
  constexpr uint32_t kIdSbf = tc::idesc_f16(128, HN, true, false, false);   // bf16 Q, K_base
  constexpr uint32_t kIdPV = tc::idesc_f16(128, D, true, false, true);
  constexpr uint32_t kIdPLV = tc::idesc_f16(128, RP, true, false, true);
  constexpr uint32_t kIdZ = tc::idesc_f16(128, D, false, false, true);  // fp16 O_lr/l x B_V

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::off_misc;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::off_misc + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::off_misc + 8 * B_COUNT + 4);
  int* stage_mask = reinterpret_cast<int*>(smem + L::off_misc + 8 * B_COUNT + 8);  // [NST]
  float2* btab = reinterpret_cast<float2*>(smem + L::off_btab);                  // [8][HALF]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s_row = blockIdx.z, head = blockIdx.y;
  const int qs = __ldg(p.q_start + s_row), qe = __ldg(p.q_start + s_row + 1);
  const int q_len = qe - qs;
  const int Ls = __ldg(p.seq_lens + s_row);
  const int g = p.g;
  const int row0 = blockIdx.x * BM;
  if (q_len <= 0 || row0 >= q_len * g) return;  // whole CTA beyond this sequence's chunk
  if (Ls < q_len || Ls > p.max_seq_len) {       // inconsistent lengths: skip, report
    if (tid == 0) report(p.status, LRKV_ERR_INDEX);
    return;
  }
  int adapter = __ldg(p.adapter_ids + s_row);
  if (adapter < -1 || adapter >= p.n_adapters) {
    if (tid == 0) report(p.status, LRKV_ERR_INDEX);
    adapter = -1;
  }
  const bool rebuild = p.has_bk && adapter >= 0;
  const bool use_lr = p.has_bv && adapter >= 0;
  const int k_first = row0 / g;
  const int k_last = min(q_len, (row0 + BM + g - 1) / g) - 1;
  const int pos_min = Ls - q_len + k_first;
  const int pos_max = Ls - q_len + k_last;
  const int U = (pos_max + HN) / HN;     // score half-tiles covering keys 0 .. pos_max
  const int n_st = (U + 1) / 2;          // stages of 128 keys

  // ---------------------------------------------------------------- setup
  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(B_FULL + i), 1);
      mbar_init(bar(B_EMPTY + i), 1);
      mbar_init(bar(B_KA + i), 128);
      mbar_init(bar(B_YFULL + i), 1);
      mbar_init(bar(B_YFREE + i), 128);
    }
    mbar_init(bar(B_SFULL + 0), 1);
    mbar_init(bar(B_SFULL + 1), 1);
    mbar_init(bar(B_PFULL + 0), 128);
    mbar_init(bar(B_PFULL + 1), 128);
    mbar_init(bar(B_OBAR), 1);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_EPI), 128);
    mbar_init(bar(B_ZFULL), 1);
    mbar_fence_init();
  }
  if (warp == 1) tc::alloc(smem_u32(tmem_slot), kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;  // this warp's TMEM lanes

  // Rebuild warpgroup state: per-row RoPE delta factors cos/sin(r * theta_j),
  // r = key % 16, packed (cos, sin) as fp16 pairs.
  uint32_t dl[HALF];
  const int rb_i = 32 * (warp & 3) + lane;  // key row (rebuild) or query row (softmax) in the tile
  if (warp >= kRbWarp0) {
    const int r = rb_i & 15;
#pragma unroll
    for (int j = 0; j < HALF; ++j) {
      const float2 cs = rope_cos_sin(r, p.freqs.hi[j], p.freqs.lo[j]);
      dl[j] = pack_f16(cs.x, cs.y);
    }
    if (rebuild) {
      // B_K^T [d][r'] (K-major, swizzled like the L_K tiles), zero beyond rank
      // R; row 32g + t holds dim 16g + t (t < 16) or d/2 + 16g + t - 16
      const __nv_bfloat16* src = p.B_K + static_cast<int64_t>(adapter) * R * p.Hkv * D + head * D;
      const int rt = tid - kRbWarp0 * 32;
      for (int e = rt; e < D * (RP / 2); e += 128) {
        const int row = e % D, k2 = e / D;
        const int t = row & 31;
        const int n = t < 16 ? 16 * (row >> 5) + t : HALF + 16 * (row >> 5) + t - 16;
        const int k0 = 2 * k2;
        const uint32_t lo = k0 < R ? __bfloat16_as_ushort(src[static_cast<int64_t>(k0) * p.Hkv * D + n]) : 0u;
        const uint32_t hi = k0 + 1 < R ? __bfloat16_as_ushort(src[static_cast<int64_t>(k0 + 1) * p.Hkv * D + n]) : 0u;
        *reinterpret_cast<uint32_t*>(smem + L::off_bk + swz<LSPAN>(row, 4 * k2)) = lo | (hi << 16);
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    }
  }
  // Softmax warpgroup: its query row into TMEM (fp16 when K_a is fp16, else bf16).
  const int sm_r = row0 + rb_i;
  const int sm_k = sm_r / g;
  const bool sm_valid = sm_k < q_len;
  const int sm_pos = Ls - q_len + (sm_valid ? sm_k : 0);
  if (warp >= kSmWarp0 && warp < kRbWarp0) {
    const __nv_bfloat16* qrow =
        p.q + (static_cast<int64_t>(qs + (sm_valid ? sm_k : 0)) * p.Hq + head * g + sm_r % g) * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t v[16];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        uint4 u = sm_valid ? __ldg(reinterpret_cast<const uint4*>(qrow + 32 * c + 8 * x)) : make_uint4(0, 0, 0, 0);
        v[4 * x + 0] = rebuild ? bf16x2_to_f16x2(u.x) : u.x;
        v[4 * x + 1] = rebuild ? bf16x2_to_f16x2(u.y) : u.y;
        v[4 * x + 2] = rebuild ? bf16x2_to_f16x2(u.z) : u.z;
        v[4 * x + 3] = rebuild ? bf16x2_to_f16x2(u.w) : u.w;
      }
      tc::st_x16(tbase + lane_off + Q_COL + 16 * c, v);
    }
    tc::wait_st();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  // ============================================================ producer
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tm_base);
      prefetch_tmap(&tm_lr);
    }
    const int nblk_vis = pos_max / kBlock + 1;  // blocks holding a key some row sees
    const uint32_t per_blk = 2u * kBlock * D * 2 + (rebuild ? kBlock * LSPAN : 0) +
                             (use_lr ? kBlock * LSPAN : 0);
    int issued = 0;
    for (int j = 0; j < n_st; ++j) {
      const int s = j % NST;
      int ok = 1;
      if (lane == 0) {
        if (*abort_flag) ok = 0;
        else if (j >= NST && !wait_phase(bar(B_EMPTY + s), ((j / NST) - 1) & 1, p.status)) ok = 0;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      int blk = -1;
      const int bi = j * 8 + lane;
      if (lane < 8 && bi < nblk_vis) {
        const int b = __ldg(p.block_tables + static_cast<int64_t>(s_row) * p.max_blocks + bi);
        if (b >= 0 && b < p.num_blocks) blk = b;
        else report(p.status, LRKV_ERR_INDEX);
      }
      const uint32_t mask = __ballot_sync(0xffffffffu, blk >= 0);
      if (lane == 0) {
        stage_mask[s] = static_cast<int>(mask);
        mbar_arrive_expect_tx(bar(B_FULL + s), __popc(mask) * per_blk);
      }
      __syncwarp();
      if (blk >= 0) {
        const uint32_t st = sbase + s * L::STAGE;
        const uint32_t fb = bar(B_FULL + s);
        const int yk = ((blk * 2 + 0) * p.Hkv + head) * kBlock;
        const int yv = ((blk * 2 + 1) * p.Hkv + head) * kBlock;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_2d(st + L::off_k + h * (BN * 128) + lane * 2048, &tm_base, 64 * h, yk, fb);
          tma_load_2d(st + L::off_v + h * (BN * 128) + lane * 2048, &tm_base, 64 * h, yv, fb);
        }
        if (rebuild) tma_load_2d(st + L::off_lk + lane * kBlock * LSPAN, &tm_lr, 0, (blk * 2 + 0) * kBlock, fb);
        if (use_lr) tma_load_2d(st + L::off_lv + lane * kBlock * LSPAN, &tm_lr, 0, (blk * 2 + 1) * kBlock, fb);
      }
      ++issued;
    }
    // after an abort, never leave copies in flight (bounded waits)
    if (lane == 0 && *abort_flag) {
      for (int j = max(0, issued - NST); j < issued; ++j)
        mbar_wait(bar(B_FULL + j % NST), (j / NST) & 1, nullptr, 1u << 16);
    }
  }

  // ================================================================= MMA
  // Fixed issue order S(0); then per half-tile u: S(u+1), P V(u). S(u+1)
  // overwrites the score buffer of u-1, whose P V was issued one step earlier
  // (MMAs execute in issue order). The whole warp runs the sequence in
  // lockstep, every decision taken from lane 0; one elected lane issues.
  if (warp == 1) {
    const uint32_t idS = rebuild ? kIdS16 : kIdSbf;
    auto uni = [&](bool c) { return __shfl_sync(0xffffffffu, static_cast<int>(c), 0) != 0; };
    auto wait_u = [&](uint32_t b, uint32_t par) { return uni(wait_phase(b, par, p.status)); };
    auto issue_S = [&](int u) {
      tc::fence_after();
      const uint32_t kt = sbase + ((u >> 1) % NST) * L::STAGE + L::off_k + (u & 1) * HN * 128;
      const uint32_t dcol = tbase + S_COL0 + 64 * (u & 1);
      if (tc::elect_one()) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t b = tc::sdesc(kt + (ks >> 2) * (BN * 128) + (ks & 3) * 32, 16, 1024, 2);
          tc::mma_ts(dcol, tbase + Q_COL + ks * 8, b, idS, ks > 0);
        }
        tc::commit(bar(B_SFULL + (u & 1)));
      }
      __syncwarp();
    };
    auto issue_PV = [&](int u) {
      tc::fence_after();
      const int s = (u >> 1) % NST;
      const uint32_t st = sbase + s * L::STAGE;
      const uint32_t pcol = tbase + S_COL0 + 64 * (u & 1);
      const uint32_t vt = st + L::off_v + (u & 1) * HN * 128;
      if (tc::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < HN / 16; ++kk) {
          const uint64_t b = tc::sdesc(vt + kk * 16 * 128, BN * 128, 1024, 2);
          tc::mma_ts(tbase + O_COL, pcol + kk * 8, b, kIdPV, (u > 0 || kk > 0) ? 1u : 0u);
        }
        if (use_lr) {
          const uint32_t lvt = st + L::off_lv + (u & 1) * HN * LSPAN;
#pragma unroll
          for (int kk = 0; kk < HN / 16; ++kk) {
            const uint64_t b = tc::sdesc(lvt + kk * 16 * LSPAN, BN * LSPAN, 8 * LSPAN, SW_LR);
            tc::mma_ts(tbase + OLR_COL, pcol + kk * 8, b, kIdPLV, (u > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc::commit(bar(B_OBAR));
        if ((u & 1) || u == U - 1) tc::commit(bar(B_EMPTY + s));
      }
      __syncwarp();
    };
    bool ok = !uni(*abort_flag != 0) && wait_u(bar(B_KA + 0), 0);
    if (ok) issue_S(0);
    for (int u = 0; ok && u < U; ++u) {
      if (u + 1 < U) {
        const int j1 = (u + 1) >> 1;
        if (!((u + 1) & 1) && !wait_u(bar(B_KA + j1 % NST), (j1 / NST) & 1)) {
          ok = false;
          break;
        }
        issue_S(u + 1);
      }
      if (!wait_u(bar(B_PFULL + (u & 1)), (u >> 1) & 1)) {
        ok = false;
        break;
      }
      issue_PV(u);
      if (uni(*abort_flag != 0)) ok = false;
    }
    if (!ok && lane == 0) *abort_flag = 1;
    // Z = fp16(O_lr / l) B_V into the score buffers (free once every P V is issued)
    if (ok && use_lr) {
      if (wait_u(bar(B_EPI), 0)) {
        tc::fence_after();
        if (tc::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < RP / 16; ++kk) {
            const uint64_t b = tc::sdesc(sbase + kk * 16 * 128, RP * 128, 1024, 2);
            tc::mma_ts(tbase + S_COL0, tbase + Q_COL + kk * 8, b, kIdZ, kk > 0);
          }
          tc::commit(bar(B_ZFULL));
        }
        __syncwarp();
      } else if (lane == 0) {
        *abort_flag = 1;
      }
    }
    // drain: every MMA issued so far completes before the tensor memory is released
    if (uni(*abort_flag != 0)) {
      if (tc::elect_one()) {
        tc::commit(bar(B_DRAIN));
        mbar_wait(bar(B_DRAIN), 0, nullptr, 1u << 16);
      }
      __syncwarp();
    }
  }

  // ============================================================ softmax
  if (warp >= kSmWarp0 && warp < kRbWarp0) {
    float m_run = -CUDART_INF_F, l_run = 0.f;
    const float sc = p.scale_log2;
    int u = 0;
    for (; u < U; ++u) {
      const int b = u & 1;
      bool ok = !*abort_flag && wait_phase(bar(B_SFULL + b), (u >> 1) & 1, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after();
      uint32_t sv[64];
      {
        uint32_t a[32], c[32];
        tc::ld_x32(tbase + lane_off + S_COL0 + 64 * b, a);
        tc::ld_x32(tbase + lane_off + S_COL0 + 64 * b + 32, c);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          sv[e] = a[e];
          sv[32 + e] = c[e];
        }
      }
      const int key0 = u * HN;
      const int bm = (stage_mask[(u >> 1) % NST] >> (4 * (u & 1))) & 0xF;
      const bool need_mask = (key0 + HN - 1 > pos_min) || bm != 0xF || !sm_valid;
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < HN; ++c) {
          const bool vis = sm_valid && (key0 + c <= sm_pos) && ((bm >> (c >> 4)) & 1);
          sv[c] = vis ? sv[c] : __float_as_uint(-CUDART_INF_F);
        }
      }
      // row max as a tree of 8 independent chains
      float mxs[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mxs[k] = __uint_as_float(sv[k]);
#pragma unroll
      for (int c = 8; c < HN; ++c) mxs[c & 7] = fmaxf(mxs[c & 7], __uint_as_float(sv[c]));
#pragma unroll
      for (int k = 0; k < 4; ++k) mxs[k] = fmaxf(mxs[k], mxs[k + 4]);
      const float mx = fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3]));
      const float mt = mx * sc;  // -inf stays -inf
      bool resc = false;
      float alpha = 1.f;
      if (mt > m_run) {
        if (m_run == -CUDART_INF_F) {
          m_run = mt;  // first visible key of this row: O and O_lr rows are still zero
        } else if (mt > m_run + kRescaleLog2) {
          alpha = ex2(m_run - mt);
          m_run = mt;
          resc = true;
        }
      }
      if (__any_sync(0xffffffffu, resc)) {
        // O and O_lr must not be in use by P V(u-1): wait for it, then rescale
        bool okw = wait_phase(bar(B_OBAR), (u - 1) & 1, p.status);
        okw = __all_sync(0xffffffffu, okw);
        if (!okw) {
          *abort_flag = 1;
          break;
        }
        tc::fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tc::ld_x32(tbase + lane_off + O_COL + 32 * c, v);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tc::st_x32(tbase + lane_off + O_COL + 32 * c, v);
        }
        if (use_lr) {
#pragma unroll
          for (int c = 0; c < RP / 16; ++c) {
            uint32_t v[16];
            tc::ld_x16(tbase + lane_off + OLR_COL + 16 * c, v);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tc::st_x16(tbase + lane_off + OLR_COL + 16 * c, v);
          }
        }
        l_run *= alpha;
      }
      uint32_t pk[32];
      float sums[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sums[k] = 0.f;
      // m_run = -inf only while no key of this row was visible: every s is -inf
      // then, and the offset 0 keeps ex2(-inf) = 0 instead of NaN
      const float moff = m_run == -CUDART_INF_F ? 0.f : m_run;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2(fmaf(__uint_as_float(sv[2 * c]), sc, -moff));
        const float p1 = ex2(fmaf(__uint_as_float(sv[2 * c + 1]), sc, -moff));
        sums[c & 7] += p0 + p1;
        pk[c] = pack_bf16(p0, p1);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) sums[k] += sums[k + 4];
      l_run += (sums[0] + sums[1]) + (sums[2] + sums[3]);
      tc::st_x32(tbase + lane_off + S_COL0 + 64 * b, pk);
      tc::wait_st();
      tc::fence_before();
      mbar_arrive(bar(B_PFULL + b));
    }
    // ---- epilogue: out = O / l + Z,  Z = fp16(O_lr / l) B_V  (one small MMA)
    bool ok = (u == U) && !*abort_flag && wait_phase(bar(B_OBAR), (U - 1) & 1, p.status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) *abort_flag = 1;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    if (ok) tc::fence_after();
    if (use_lr) {
      if (ok) {
        // B_V [R][d] -> fp16, MN-major with 128-byte swizzle, into stage 0 (idle:
        // every MMA has completed); rows R .. r'-1 are zero
        const __nv_bfloat16* src = p.B_V + static_cast<int64_t>(adapter) * R * p.Hkv * D + head * D;
        for (int e = rb_i; e < RP * (D / 8); e += 128) {
          const int k = e / (D / 8), v8 = e % (D / 8);
          uint4 w = make_uint4(0, 0, 0, 0);
          if (k < R) {
            w = __ldg(reinterpret_cast<const uint4*>(src + static_cast<int64_t>(k) * p.Hkv * D) + v8);
            w.x = bf16x2_to_f16x2(w.x);
            w.y = bf16x2_to_f16x2(w.y);
            w.z = bf16x2_to_f16x2(w.z);
            w.w = bf16x2_to_f16x2(w.w);
          }
          *reinterpret_cast<uint4*>(smem + (v8 / 8) * (RP * 128) + swz<128>(k, (v8 % 8) * 16)) = w;
        }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        // fp16(O_lr / l) as the A operand, over the (no longer needed) Q columns
#pragma unroll
        for (int c = 0; c < RP / 32 + (RP % 32 ? 1 : 0); ++c) {
          uint32_t v[16];
          uint32_t f[16];
          tc::ld_x16(tbase + lane_off + OLR_COL + 32 * c, v);
          if (RP - 32 * c > 16) tc::ld_x16(tbase + lane_off + OLR_COL + 32 * c + 16, f);
          tc::wait_ld();
          uint32_t a[16];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            a[e] = pack_f16(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            a[8 + e] = (RP - 32 * c > 16) ? pack_f16(__uint_as_float(f[2 * e]) * inv, __uint_as_float(f[2 * e + 1]) * inv) : 0u;
          tc::st_x16(tbase + lane_off + Q_COL + 16 * c, a);
        }
        tc::wait_st();
        tc::fence_before();
      }
      mbar_arrive(bar(B_EPI));
      bool okz = ok && wait_phase(bar(B_ZFULL), 0, p.status);
      okz = __all_sync(0xffffffffu, okz);
      if (!okz) *abort_flag = 1;
      ok = okz;
      if (ok) tc::fence_after();
    }
    if (ok) {
      __nv_bfloat16* orow = p.out + (static_cast<int64_t>(qs + (sm_valid ? sm_k : 0)) * p.Hq + head * g + sm_r % g) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32], z[32];
        tc::ld_x32(tbase + lane_off + O_COL + 32 * c, v);
        if (use_lr) tc::ld_x32(tbase + lane_off + S_COL0 + 32 * c, z);
        tc::wait_ld();
        if (sm_valid) {
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o[e] = __uint_as_float(v[8 * x + e]) * inv + (use_lr ? __uint_as_float(z[8 * x + e]) : 0.f);
            uint4 w;
            w.x = pack_bf16(o[0], o[1]);
            w.y = pack_bf16(o[2], o[3]);
            w.z = pack_bf16(o[4], o[5]);
            w.w = pack_bf16(o[6], o[7]);
            *reinterpret_cast<uint4*>(orow + 32 * c + 8 * x) = w;
          }
        }
      }
    }
  }

  // ============================================================ rebuild
  if (warp >= kRbWarp0) {
    const int i = rb_i;       // key row within the stage
    const int bb = i >> 4;    // block within the stage
    // Every exit from this loop is decided by a barrier vote of the whole
    // warpgroup (bar.red.or), so no warp is left waiting at a named barrier;
    // a warp whose wait failed skips its work until the next vote.
    // The warpgroup issues its own Y MMAs (one elected lane of its first
    // warp; commits track each issuing thread separately): Y(j+1) as soon as
    // every thread has read Y(j) and stage j+1 has landed, else right after
    // stage j+1's tiles are seen.
    bool failed = false;
    bool y_next = false;  // Y of the coming stage already issued (issuing warp only)
    const bool y_warp = warp == kRbWarp0;
    auto issue_Y = [&](int jj) {
      tc::fence_after();
      const uint32_t stj = sbase + (jj % NST) * L::STAGE;
      if (tc::elect_one()) {
#pragma unroll
        for (int gy = 0; gy < NG; ++gy) {
#pragma unroll
          for (int kk = 0; kk < RP / 16; ++kk) {
            const uint64_t a = tc::sdesc(stj + L::off_lk + kk * 32, 16, 8 * LSPAN, SW_LR);
            const uint64_t b = tc::sdesc(sbase + L::off_bk + 32 * gy * LSPAN + kk * 32, 16, 8 * LSPAN, SW_LR);
            tc::mma_ss(tbase + Y_COL + 32 * gy, a, b, kIdY, kk > 0);
          }
          tc::commit(bar(B_YFULL + gy));
        }
      }
      __syncwarp();
    };
    for (int j = 0; j < n_st; ++j) {
      const int s = j % NST;
      const uint32_t st = sbase + s * L::STAGE;
      // the previous stage's readers of btab are done past this barrier
      if (named_bar_or(3, 128, failed || *abort_flag != 0)) break;
      if (rebuild) {  // block start angles of this stage
        for (int e = i; e < 8 * HALF; e += 128) {
          const int b2 = e / HALF, jj = e % HALF;
          btab[e] = rope_cos_sin_fast(j * BN + kBlock * b2, p.freqs.hi[jj], p.freqs.lo[jj]);
        }
      }
      failed = !wait_phase(bar(B_FULL + s), (j / NST) & 1, p.status);
      if (named_bar_or(3, 128, failed)) {  // also publishes btab to the warpgroup
        *abort_flag = 1;
        break;
      }
      const int mask = stage_mask[s];
      const int t = j * BN + i;
      const bool key_ok = ((mask >> bb) & 1) && t < Ls;
      if (rebuild) {
        if (y_warp && !y_next) issue_Y(j);
        const float2* bt = btab + bb * HALF;
#pragma unroll
        for (int grp = 0; grp < NG; ++grp) {
          bool oky = !failed && wait_phase(bar(B_YFULL + grp), j & 1, p.status);
          oky = __all_sync(0xffffffffu, oky);
          if (!oky) {
            failed = true;
            *abort_flag = 1;
          }
          if (failed) continue;
          tc::fence_after();
          uint32_t y[32];  // [0, 16): dims 16 grp + e; [16, 32): their partners
          tc::ld_x32(tbase + lane_off + Y_COL + 32 * grp, y);
          tc::wait_ld();
          if (key_ok) {
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {  // 8 pairs per 16-byte chunk
              const int dlo = 16 * grp + 8 * hc, dhi = dlo + HALF;
              const uint32_t alo = st + L::off_k + (dlo / 64) * (BN * 128) + swz<128>(i, (dlo % 64) * 2);
              const uint32_t ahi = st + L::off_k + (dhi / 64) * (BN * 128) + swz<128>(i, (dhi % 64) * 2);
              uint4 klo, khi;
              asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                           : "=r"(klo.x), "=r"(klo.y), "=r"(klo.z), "=r"(klo.w) : "r"(alo));
              asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                           : "=r"(khi.x), "=r"(khi.y), "=r"(khi.z), "=r"(khi.w) : "r"(ahi));
              const uint32_t kl[4] = {klo.x, klo.y, klo.z, klo.w};
              const uint32_t kh[4] = {khi.x, khi.y, khi.z, khi.w};
              uint32_t olo[4], ohi[4];
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                float rl[2], rh[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int pp = 8 * hc + 2 * w + e;  // pair index within the group
                  const int jj = 16 * grp + pp;
                  const float2 b2 = bt[jj];
                  const float cd = __half2float(__ushort_as_half(static_cast<unsigned short>(dl[jj] & 0xffffu)));
                  const float sd = __half2float(__ushort_as_half(static_cast<unsigned short>(dl[jj] >> 16)));
                  const float c = b2.x * cd - b2.y * sd;
                  const float sn = b2.y * cd + b2.x * sd;
                  const float yl = __uint_as_float(y[pp]), yh = __uint_as_float(y[16 + pp]);
                  const float bl = e ? bf16_hi(kl[w]) : bf16_lo(kl[w]);
                  const float bh = e ? bf16_hi(kh[w]) : bf16_lo(kh[w]);
                  rl[e] = fmaf(yl, c, fmaf(-yh, sn, bl));
                  rh[e] = fmaf(yh, c, fmaf(yl, sn, bh));
                }
                olo[w] = pack_f16(rl[0], rl[1]);
                ohi[w] = pack_f16(rh[0], rh[1]);
              }
              asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(alo), "r"(olo[0]), "r"(olo[1]),
                           "r"(olo[2]), "r"(olo[3]) : "memory");
              asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(ahi), "r"(ohi[0]), "r"(ohi[1]),
                           "r"(ohi[2]), "r"(ohi[3]) : "memory");
            }
          }
        }
        // every thread has read Y(j): issue Y(j+1) now if its tiles are there
        tc::fence_before();
        if (named_bar_or(3, 128, failed)) {
          *abort_flag = 1;
          break;
        }
        y_next = false;
        if (y_warp && j + 1 < n_st &&
            __shfl_sync(0xffffffffu, static_cast<int>(test_parity(bar(B_FULL + (j + 1) % NST), ((j + 1) / NST) & 1)), 0)) {
          issue_Y(j + 1);
          y_next = true;
        }
      }
      if (failed) continue;
      // Keys past the sequence end or in a block that was not loaded: zero their
      // V and L_V rows, so that P = 0 there cannot meet stale (NaN) data.
      if (!key_ok) {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint32_t a = st + L::off_v + (c / 8) * (BN * 128) + swz<128>(i, (c % 8) * 16);
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(a), "r"(0u) : "memory");
        }
        if (use_lr) {
#pragma unroll
          for (int c = 0; c < LSPAN / 16; ++c) {
            const uint32_t a = st + L::off_lv + swz<LSPAN>(i, c * 16);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(a), "r"(0u) : "memory");
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      mbar_arrive(bar(B_KA + s));
    }
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tbase, kTmemCols);
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
  CUtensorMap tb, tl;
  if (!make_pool_maps(cfg, a.base_pool, a.lr_pool, a.num_blocks, &tb, nullptr)) return LRKV_ERR_CUDA;
  if (!make_lr_map(cfg, a.lr_pool, a.num_blocks, PL<D, R>::RP, &tl)) return LRKV_ERR_CUDA;
  auto kern = prefill_kernel<D, R>;
  constexpr int smem = PL<D, R>::total;
  static bool attr_set = false;  // idempotent per-process kernel attribute
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return LRKV_ERR_CUDA;
    attr_set = true;
  }
  const int tiles = (a.max_q_len * p.g + BM - 1) / BM;
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
