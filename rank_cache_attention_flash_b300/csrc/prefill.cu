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
// share every key tile. Per tile of BN keys (BN / 16 paged blocks):
//   Y         = L_K B_K               tcgen05 (rebuild warpgroup)   -> TMEM
//   K_a       = K_base + RoPE(Y)      rebuild warpgroup, in place in the tile's
//                                     K buffer (fp16, never stored to HBM)
//   S         = Q K_a^T               tcgen05, Q read from TMEM       -> TMEM
//   P         = online softmax(S)     softmax warpgroup, thread = query row,
//                                     P (bf16) to its own TMEM columns
//   O += P V_base, O_lr += P L_V      tcgen05, P read from TMEM
// and at the end out = O / l + fp16(O_lr / l) B_V (one more small MMA).
//
// A tcgen05.mma takes about as long to issue from one warp as the tensor
// pipe needs for a 128 x 192 x 16 product, so every MMA is made as wide as
// the data allows and the independent streams are issued by different
// warps: S by warp 1, P V by warp 2, P L_V by warp 3, Y by the rebuild
// warpgroup. Y is produced in quarters of 16 RoPE pairs (B_K^T is staged
// with its rows in that order) into two TMEM buffers, so the next quarters
// compute while the current one is rotated.
// Warp roles (512 threads): warp 0 streams K, V, L_V, L_K tiles with 2-D TMA
// copies into an mbarrier ring; warp 1 owns the tensor memory and issues S;
// warps 2 and 3 issue P V and P L_V; warps 4-7 run the softmax; warps 8-11
// rebuild K_a; warp 12 issues Y (warps 13-15 only take part in the barriers). Tensor-memory columns: Q [0, d/2) (packed 16-bit),
// S [64, 64 + BN), P [192, 192 + BN/2) (packed bf16), O [256, 256 + d),
// O_lr [256 + d, 256 + d + r'), Y [448, 512) (two buffers of 32 columns).
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

constexpr int kThreads = 512;
constexpr int BM = 128;  // query rows per CTA (= TMEM lanes)
constexpr int kSmemLimit = 227 * 1024;
constexpr uint32_t kTmemCols = 512;
constexpr int Q_COL = 0, S_COL = 64, P_COL = 192, O_COL = 256, Y_COL = 448;
constexpr int kSmWarp0 = 4, kRbWarp0 = 8;  // first softmax / rebuild warp
constexpr float kRescaleLog2 = 8.0f;       // rescale O only when the row max grows by > 2^8
constexpr int kYWarp = 12;                 // Y issuer (warps 13-15 idle)
constexpr int kLaunchRegs = 128;           // 65536 / 512
constexpr int kLowRegs = 40, kHighRegs = 216;
static_assert(256 * kLowRegs + 256 * kHighRegs == kThreads * kLaunchRegs, "register split");

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
  int lr_groups;  // > 1: agent-specific A, adapter a's low-rank group at columns [a r, (a+1) r)
  int has_bk, has_bv;
  float scale_log2;
  const uint8_t* cbase;  // compressed base pool (CODEC kernels): chunks of codec_chunk_bytes(D)
  float vcent[8];        // value-code centroids (Lloyd-Max for N(0,1)), ascending
  RopeFreqs freqs;
};

// Shared-memory layout (byte offsets from a 1024-aligned base). A stage holds
// one key tile: K (rebuilt in place), V, L_V, L_K. The tile is the widest
// multiple of 16 keys up to 128 that leaves room for three stages.
constexpr int pl_stage(int D, int R, int bn) { return 2 * bn * D * 2 + 2 * bn * (R < 16 ? 32 : 2 * R); }
constexpr int pl_fixed(int D, int R, int bn) {
  return D * (R < 16 ? 32 : 2 * R) + (bn / 16) * (D / 2) * 8 + 16 * ((D / 2) * 8 + 16) + 512 + 1024;
}
constexpr int pl_bn(int D, int R) {
  int bn = 128;
  while (bn > 64 && (kSmemLimit - pl_fixed(D, R, bn)) / pl_stage(D, R, bn) < 3) bn -= 16;
  return bn;
}
template <int D, int R>
struct PL {
  static constexpr int RP = R < 16 ? 16 : R;      // rank padded to the MMA granularity
  static constexpr int LSPAN = RP * 2;            // bytes per low-rank row (32 / 64 / 128)
  static constexpr int BN = pl_bn(D, R);          // keys per tile
  static constexpr int NB = BN / 16;              // paged blocks per tile
  static constexpr int KV = BN * D * 2;           // K or V tile
  static constexpr int LT = BN * LSPAN;           // L_V or L_K tile
  static constexpr int STAGE = 2 * KV + 2 * LT;
  static constexpr int BKB = D * LSPAN;           // B_K^T tile [d][r'], K-major
  static constexpr int BTAB = NB * (D / 2) * 8;   // per-tile block start angles (cos, sin)
  static constexpr int DPITCH = (D / 2) * 8 + 16; // delta-table row: d/2 (cos, sin) + pad
  static constexpr int DTAB = 16 * DPITCH;        // cos / sin(r theta_j), r < 16
  static constexpr int MISC = 512;
  static constexpr int FIXED = BKB + BTAB + DTAB + MISC + 1024;
  static constexpr int NST_FIT = (kSmemLimit - FIXED) / STAGE;
  static constexpr int NST = NST_FIT > 4 ? 4 : NST_FIT;
  static constexpr int off_k = 0, off_v = KV, off_lv = 2 * KV, off_lk = 2 * KV + LT;
  static constexpr int off_bk = NST * STAGE;
  static constexpr int off_btab = off_bk + BKB;
  static constexpr int off_dtab = off_btab + BTAB;
  static constexpr int off_misc = off_dtab + DTAB;
  static_assert(FIXED == pl_fixed(D, R, BN) && STAGE == pl_stage(D, R, BN), "layout");
  static_assert(KV % 1024 == 0 && LT % 256 == 0 && (2 * KV + LT) % (8 * LSPAN) == 0, "atom alignment");
  static constexpr int total = off_misc + MISC + 1024;  // + alignment slack
  static_assert(NST >= 2, "two pipeline stages must fit");
  static_assert(total <= kSmemLimit, "shared memory");
  static_assert(S_COL + BN <= P_COL && P_COL + BN / 2 <= O_COL && O_COL + D + RP <= Y_COL &&
                    Y_COL + 64 <= 512, "tensor-memory columns");

  static_assert(RP * D * 2 <= KV, "B_V staging fits the first K buffer");
};

// Barrier slots inside the misc area (8 bytes each).
enum : int {
  B_FULL = 0,    // [4] TMA -> consumers (one phase per stage use)
  B_EMPTY = 4,   // [4] P V and P L_V issuer commits -> producer
  B_KA = 8,      // [4] rebuild warpgroup -> S issuer (K_a written)
  B_YFULL = 24,  // [2] Y issuer commit -> rebuild warpgroup (per Y buffer)
  B_YFREE = 26,  // [2] rebuild warpgroup -> Y issuer (quarter read from the buffer)
  B_SFULL = 13,  // S issuer commit -> softmax
  B_SFREE = 14,  // softmax -> S issuer (S loaded into registers)
  B_PFULL = 15,  // softmax -> P V / P L_V issuers (P in TMEM, O rescaled)
  B_OBAR = 16,   // P V issuer commit after each tile
  B_LBAR = 17,   // P L_V issuer commit after each tile
  B_EPI = 18,    // softmax -> P V issuer: fp16(O_lr / l) in TMEM, B_V in smem
  B_ZFULL = 19,  // P V issuer commit -> softmax
  B_DRAIN = 20,  // [4] per issuer, on abort: every MMA it issued has completed
  B_COUNT = 28
};

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

constexpr long long kWaitCycles = 1ll << 31;  // ~1 s: a wait this long has failed

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

// 2^x by the hardware approximation (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

template <int D, int R, bool CODEC>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p,
                   const __grid_constant__ CUtensorMap tm_base,
                   const __grid_constant__ CUtensorMap tm_lk,
                   const __grid_constant__ CUtensorMap tm_base_run,
                   const __grid_constant__ CUtensorMap tm_lr_run) {
  using L = PL<D, R>;
  constexpr int HALF = D / 2;
  constexpr int RP = L::RP;
  constexpr int LSPAN = L::LSPAN;
  constexpr int NST = L::NST;
  constexpr int BN = L::BN;
  constexpr int NB = L::NB;
  constexpr uint32_t SW_LK = tc::swizzle_code(LSPAN);
  constexpr int NQ = HALF / 16;  // Y quarters of 16 RoPE pairs per tile
  static_assert(NQ % 2 == 0, "the rebuild takes the quarters in pairs");
  constexpr uint32_t kIdY = tc::idesc_f16(128, 32, true, false, false);
  constexpr uint32_t kIdS16 = tc::idesc_f16(128, BN, false, false, false);  // fp16 Q, K_a
  constexpr uint32_t kIdSbf = tc::idesc_f16(128, BN, true, false, false);   // bf16 Q, K_base
  constexpr uint32_t kIdPV = tc::idesc_f16(128, D, true, false, true);
  constexpr uint32_t kIdPLV = tc::idesc_f16(128, RP, true, false, true);
  constexpr uint32_t kIdZ = tc::idesc_f16(128, D, false, false, true);  // fp16 O_lr/l x B_V

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, offset from the shared array itself so that the
  // compiler keeps every access through it in the shared address space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::off_misc;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::off_misc + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::off_misc + 8 * B_COUNT + 4);
  int* stage_mask = reinterpret_cast<int*>(smem + L::off_misc + 8 * B_COUNT + 8);  // [NST]
  float2* btab = reinterpret_cast<float2*>(smem + L::off_btab);                  // [NB][HALF]

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
  // compressed base pool: the rebuild warpgroup expands each tile's key codes
  // to fp16 (scored in fp16 like a rebuilt K_a) and its value codes to bf16 in
  // the rotated domain; the epilogue rotates the output back
  const bool kconv = rebuild || CODEC;
  // agent-specific A: this sequence's adapter reads its own low-rank group
  const int lr_x = (p.lr_groups > 1 && adapter >= 0) ? adapter * R : 0;
  const int k_first = row0 / g;
  const int k_last = min(q_len, (row0 + BM + g - 1) / g) - 1;
  const int pos_min = Ls - q_len + k_first;
  const int pos_max = Ls - q_len + k_last;
  const int U = (pos_max + BN) / BN;  // key tiles covering keys 0 .. pos_max

  // ---------------------------------------------------------------- setup
  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(B_FULL + i), 1);
      mbar_init(bar(B_EMPTY + i), use_lr ? 2 : 1);
      mbar_init(bar(B_KA + i), 128);
      mbar_init(bar(B_DRAIN + i), 1);
    }
    mbar_init(bar(B_YFULL + 0), 1);
    mbar_init(bar(B_YFULL + 1), 1);
    mbar_init(bar(B_YFREE + 0), 128);
    mbar_init(bar(B_YFREE + 1), 128);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_SFREE), 128);
    mbar_init(bar(B_PFULL), 128);
    mbar_init(bar(B_OBAR), 1);
    mbar_init(bar(B_LBAR), 1);
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
  const int rb_i = 32 * (warp & 3) + lane;  // key row (rebuild) or query row (softmax) in the tile

  // Rebuild warpgroup: B_K^T staged in smem (the RoPE delta factors are set
  // up once the warpgroup has its larger register share, below).
  if (warp >= kRbWarp0) {
    if (rebuild) {
      // B_K^T [d][r'] (K-major, swizzled like the L_K tiles), zero beyond rank
      // R; row 32 q + t holds dim 16 q + t (t < 16) or d/2 + 16 q + t - 16
      const __nv_bfloat16* src = p.B_K + static_cast<int64_t>(adapter) * R * p.Hkv * D + head * D;
      for (int e = rb_i; e < D * (RP / 2); e += 128) {
        const int row = e % D, k2 = e / D;
        const int q = row / 32, t = row % 32;
        const int n = t < 16 ? 16 * q + t : HALF + 16 * q + t - 16;
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
        v[4 * x + 0] = kconv ? bf16x2_to_f16x2(u.x) : u.x;
        v[4 * x + 1] = kconv ? bf16x2_to_f16x2(u.y) : u.y;
        v[4 * x + 2] = kconv ? bf16x2_to_f16x2(u.z) : u.z;
        v[4 * x + 3] = kconv ? bf16x2_to_f16x2(u.w) : u.w;
      }
      tc::st_x16(tbase + lane_off + Q_COL + 16 * c, v);
    }
    tc::wait_st();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  // Register split: the launch gives every thread kLaunchRegs; warpgroups 0
  // and 3 (producer, MMA issuers, Y issuer) hand registers to the softmax and
  // rebuild warpgroups (256 * kLowRegs + 256 * kHighRegs = 512 * kLaunchRegs),
  // each warpgroup at the top of its own branch below.
  auto uni = [&](bool c) { return __shfl_sync(0xffffffffu, static_cast<int>(c), 0) != 0; };

  if (warp < kSmWarp0) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kLowRegs));
  // ============================================================ producer
  if (warp == 0) {
    if (lane == 0) {
      if (!CODEC) prefetch_tmap(&tm_base);
      prefetch_tmap(&tm_lk);
      if (!CODEC) {
        prefetch_tmap(&tm_base_run);
        prefetch_tmap(&tm_lr_run);
      }
    }
    const int nblk_vis = pos_max / kBlock + 1;  // blocks holding a key some row sees
    // per block: K and V (planes, or the compressed chunk's Kq|Ks and Vq|Vn), L_V, L_K
    const uint32_t base_blk = CODEC ? codec_k_bytes(D) + codec_v_bytes(D) : 2u * kBlock * D * 2;
    const uint32_t per_blk = base_blk + (use_lr ? kBlock * LSPAN : 0) + (rebuild ? kBlock * LSPAN : 0);
    const int32_t* bt_row = p.block_tables + static_cast<int64_t>(s_row) * p.max_blocks;
    // block ids of the next tile are fetched one tile ahead (lane b: block b)
    int id_next = (lane < NB && lane < nblk_vis) ? __ldg(bt_row + lane) : -1;
    int issued = 0;
    for (int j = 0; j < U; ++j) {
      const int s = j % NST;
      const int id = id_next;
      const int bn = (j + 1) * NB + lane;
      id_next = (lane < NB && bn < nblk_vis) ? __ldg(bt_row + bn) : -1;
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
      if (lane < NB && j * NB + lane < nblk_vis) {
        if (id >= 0 && id < p.num_blocks) blk = id;
        else report(p.status, LRKV_ERR_INDEX);
      }
      const uint32_t mask = __ballot_sync(0xffffffffu, blk >= 0);
      // one copy per plane when the tile's blocks are consecutive in the pool
      const int blk0 = __shfl_sync(0xffffffffu, blk, 0);
      const bool run = !CODEC && mask == (1u << NB) - 1 && __all_sync(0xffffffffu, lane >= NB || blk == blk0 + lane);
      if (lane == 0) {
        stage_mask[s] = static_cast<int>(mask);
        mbar_arrive_expect_tx(bar(B_FULL + s), __popc(mask) * per_blk);
      }
      __syncwarp();
      const uint32_t st = sbase + s * L::STAGE;
      const uint32_t fb = bar(B_FULL + s);
      if (run) {
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_4d(st + L::off_k + h * (BN * 128), &tm_base_run, 64 * h, 0, head, blk0, fb);
            tma_load_4d(st + L::off_v + h * (BN * 128), &tm_base_run, 64 * h, 0, p.Hkv + head, blk0, fb);
          }
          if (use_lr) tma_load_4d(st + L::off_lv, &tm_lr_run, lr_x, 0, 1, blk0, fb);
          if (rebuild) tma_load_4d(st + L::off_lk, &tm_lr_run, lr_x, 0, 0, blk0, fb);
        }
      } else if (blk >= 0) {
        if (CODEC) {
          // the block's codes, staged at the front of the tile's K and V buffers
          const uint8_t* chunk = p.cbase + (static_cast<int64_t>(blk) * p.Hkv + head) * codec_chunk_bytes(D);
          bulk_load(st + L::off_k + lane * codec_k_bytes(D), chunk, codec_k_bytes(D), fb);
          bulk_load(st + L::off_v + lane * codec_v_bytes(D), chunk + codec_k_bytes(D), codec_v_bytes(D), fb);
        } else {
          const int yk = ((blk * 2 + 0) * p.Hkv + head) * kBlock;
          const int yv = ((blk * 2 + 1) * p.Hkv + head) * kBlock;
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_2d(st + L::off_k + h * (BN * 128) + lane * 2048, &tm_base, 64 * h, yk, fb);
            tma_load_2d(st + L::off_v + h * (BN * 128) + lane * 2048, &tm_base, 64 * h, yv, fb);
          }
        }
        if (use_lr) tma_load_2d(st + L::off_lv + lane * kBlock * LSPAN, &tm_lk, lr_x, (blk * 2 + 1) * kBlock, fb);
        if (rebuild) tma_load_2d(st + L::off_lk + lane * kBlock * LSPAN, &tm_lk, lr_x, (blk * 2 + 0) * kBlock, fb);
      }
      ++issued;
    }
    // after an abort, never leave copies in flight (bounded waits)
    if (lane == 0 && *abort_flag) {
      for (int j = max(0, issued - NST); j < issued; ++j)
        mbar_wait(bar(B_FULL + j % NST), (j / NST) & 1, nullptr, 1u << 16);
    }
  }

  // ============================================================ S issuer
  // S(u) = Q K_a(u)^T into the single score buffer, once the rebuild has
  // written K_a(u) and the softmax has loaded S(u-1).
  if (warp == 1) {
    const uint32_t idS = kconv ? kIdS16 : kIdSbf;
    const uint64_t bdesc0 = tc::sdesc(sbase + L::off_k, 16, 1024, 2);
    bool ok = true;
    for (int u = 0; u < U; ++u) {
      const int s = u % NST;
      if (uni(*abort_flag != 0) || !uni(wait_phase(bar(B_KA + s), (u / NST) & 1, p.status)) ||
          (u > 0 && !uni(wait_phase(bar(B_SFREE), (u - 1) & 1, p.status)))) {
        ok = false;
        break;
      }
      tc::fence_after();
      if (tc::elect_one()) {
        const uint64_t bd = bdesc0 + ((s * L::STAGE) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc::mma_ts(tbase + S_COL, tbase + Q_COL + ks * 8, bd + (((ks >> 2) * (BN * 128) + (ks & 3) * 32) >> 4),
                     idS, ks > 0);
        tc::commit(bar(B_SFULL));
      }
      __syncwarp();
    }
    if (!ok && lane == 0) *abort_flag = 1;
    if (uni(*abort_flag != 0)) {
      if (tc::elect_one()) {
        tc::commit(bar(B_DRAIN + 1));
        mbar_wait(bar(B_DRAIN + 1), 0, nullptr, 1u << 16);
      }
      __syncwarp();
    }
  }

  // ================================================== P V / P L_V issuers
  // O += P(u) V (warp 2) and O_lr += P(u) L_V (warp 3) once the softmax has
  // written P(u); each commit releases the stage (two arrivals when both run).
  // At the end warp 2 also computes Z = fp16(O_lr / l) B_V.
  if (warp == 2 || (warp == 3 && use_lr)) {
    const bool lv = warp == 3;
    const uint64_t bdesc0 = lv ? tc::sdesc(sbase + L::off_lv, BN * LSPAN, 8 * LSPAN, SW_LK)
                               : tc::sdesc(sbase + L::off_v, BN * 128, 1024, 2);
    const uint32_t dcol = tbase + (lv ? O_COL + D : O_COL);
    const uint32_t idPV = lv ? kIdPLV : kIdPV;
    const uint32_t row_bytes = lv ? LSPAN : 128;
    bool ok = true;
    for (int u = 0; u < U; ++u) {
      const int s = u % NST;
      if (uni(*abort_flag != 0) || !uni(wait_phase(bar(B_PFULL), u & 1, p.status))) {
        ok = false;
        break;
      }
      tc::fence_after();
      if (tc::elect_one()) {
        const uint64_t bd = bdesc0 + ((s * L::STAGE) >> 4);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          tc::mma_ts(dcol, tbase + P_COL + kk * 8, bd + ((kk * 16 * row_bytes) >> 4), idPV,
                     (u > 0 || kk > 0) ? 1u : 0u);
        tc::commit(bar(lv ? B_LBAR : B_OBAR));
        tc::commit(bar(B_EMPTY + s));
      }
      __syncwarp();
    }
    if (!ok && lane == 0) *abort_flag = 1;
    if (!lv && ok && use_lr) {
      if (uni(wait_phase(bar(B_EPI), 0, p.status))) {
        tc::fence_after();
        if (tc::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < RP / 16; ++kk) {
            const uint64_t b = tc::sdesc(sbase + kk * 16 * 128, RP * 128, 1024, 2);
            tc::mma_ts(tbase + S_COL, tbase + Q_COL + kk * 8, b, kIdZ, kk > 0);
          }
          tc::commit(bar(B_ZFULL));
        }
        __syncwarp();
      } else if (lane == 0) {
        *abort_flag = 1;
      }
    }
    if (uni(*abort_flag != 0)) {
      if (tc::elect_one()) {
        tc::commit(bar(B_DRAIN + warp));
        mbar_wait(bar(B_DRAIN + warp), 0, nullptr, 1u << 16);
      }
      __syncwarp();
    }
  }
  }  // warpgroup 0
  // ============================================================ softmax
  else if (warp < kRbWarp0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kHighRegs));
    float m_run = -CUDART_INF_F, l_run = 0.f;
    const float sc = p.scale_log2;
    int u = 0;
    for (; u < U; ++u) {
      bool ok = !*abort_flag && wait_phase(bar(B_SFULL), u & 1, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after();
      uint32_t sv[BN];
#pragma unroll
      for (int c = 0; c < BN / 16; ++c) {
        uint32_t a[16];
        tc::ld_x16(tbase + lane_off + S_COL + 16 * c, a);
#pragma unroll
        for (int e = 0; e < 16; ++e) sv[16 * c + e] = a[e];
      }
      tc::wait_ld();
      tc::fence_before();
      mbar_arrive(bar(B_SFREE));  // the score buffer may take S(u+1)
      const int key0 = u * BN;
      const int bm = stage_mask[u % NST];
      const bool need_mask = (key0 + BN - 1 > pos_min) || bm != (1 << NB) - 1 || !sm_valid;
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const bool vis = sm_valid && (key0 + c <= sm_pos) && ((bm >> (c >> 4)) & 1);
          sv[c] = vis ? sv[c] : __float_as_uint(-CUDART_INF_F);
        }
      }
      // row max as a tree of 8 independent chains
      float mxs[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mxs[k] = __uint_as_float(sv[k]);
#pragma unroll
      for (int c = 8; c < BN; ++c) mxs[c & 7] = fmaxf(mxs[c & 7], __uint_as_float(sv[c]));
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
      // P(u-1) V and P(u-1) L_V must have completed: they read the P columns
      // and write O, O_lr
      if (u > 0) {
        bool okw = wait_phase(bar(B_OBAR), (u - 1) & 1, p.status);
        if (use_lr) okw = okw && wait_phase(bar(B_LBAR), (u - 1) & 1, p.status);
        okw = __all_sync(0xffffffffu, okw);
        if (!okw) {
          *abort_flag = 1;
          break;
        }
        tc::fence_after();
      }
      if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int c = 0; c < (D + RP + 31) / 32; ++c) {
          uint32_t v[32];
          tc::ld_x32(tbase + lane_off + O_COL + 32 * c, v);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tc::st_x32(tbase + lane_off + O_COL + 32 * c, v);
        }
        l_run *= alpha;
      }
      // P = 2^(s * scale - m) as packed bf16 into the P columns of this row
      float sums[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sums[k] = 0.f;
      // m_run = -inf only while no key of this row was visible: every s is -inf
      // then, and the offset 0 keeps ex2(-inf) = 0 instead of NaN
      const float moff = m_run == -CUDART_INF_F ? 0.f : m_run;
#pragma unroll
      for (int c16 = 0; c16 < BN / 16; ++c16) {
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float p0 = ex2(fmaf(__uint_as_float(sv[16 * c16 + 2 * e]), sc, -moff));
          const float p1 = ex2(fmaf(__uint_as_float(sv[16 * c16 + 2 * e + 1]), sc, -moff));
          sums[e] += p0 + p1;
          w[e] = pack_bf16(p0, p1);
        }
        tc::st_x8(tbase + lane_off + P_COL + 8 * c16, w);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) sums[k] += sums[k + 4];
      l_run += (sums[0] + sums[1]) + (sums[2] + sums[3]);
      tc::wait_st();
      tc::fence_before();
      mbar_arrive(bar(B_PFULL));
    }
    // ---- epilogue: out = O / l + Z,  Z = fp16(O_lr / l) B_V  (one small MMA)
    bool ok = (u == U) && !*abort_flag && wait_phase(bar(B_OBAR), (U - 1) & 1, p.status) &&
              (!use_lr || wait_phase(bar(B_LBAR), (U - 1) & 1, p.status));
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) *abort_flag = 1;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    if (ok) tc::fence_after();
    if (use_lr) {
      if (ok) {
        // B_V [R][d] -> fp16, MN-major with 128-byte swizzle, into stage 0's K
        // buffer (idle: every MMA has completed); rows R .. r'-1 are zero
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
        for (int c = 0; c < (RP + 31) / 32; ++c) {
          uint32_t v[16];
          uint32_t f[16];
          tc::ld_x16(tbase + lane_off + O_COL + D + 32 * c, v);
          if (RP - 32 * c > 16) tc::ld_x16(tbase + lane_off + O_COL + D + 32 * c + 16, f);
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
        if (CODEC) {
          // O_base = (H / sqrt(d)) O_rot: group c of H O_rot is fwht32 of
          // sum_k (-1)^popc(c & k) O_rot[32 k ..]
          float zr[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) zr[e] = 0.f;
#pragma unroll
          for (int k = 0; k < D / 32; ++k) {
            uint32_t x[32];
            tc::ld_x32(tbase + lane_off + O_COL + 32 * k, x);
            tc::wait_ld();
            const bool neg = (__popc(c & k) & 1) != 0;
#pragma unroll
            for (int e = 0; e < 32; ++e) zr[e] += neg ? -__uint_as_float(x[e]) : __uint_as_float(x[e]);
          }
          fwht32(zr);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(zr[e] * (1.0f / kSqrtD<D>));
        } else {
          tc::ld_x32(tbase + lane_off + O_COL + 32 * c, v);
        }
        if (use_lr) tc::ld_x32(tbase + lane_off + S_COL + 32 * c, z);
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
  else if (warp < kYWarp) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kHighRegs));
    // RoPE delta table cos / sin(r * theta_j), r < 16, in smem (padded rows:
    // the 16 rows a warp reads at once fall in distinct banks); kept out of
    // registers so that the rotation loop stays rolled (small code)
    for (int e = rb_i; e < 16 * HALF; e += 128) {
      const int r = e / HALF, j = e % HALF;
      *reinterpret_cast<float2*>(smem + L::off_dtab + r * L::DPITCH + j * 8) =
          rope_cos_sin(r, p.freqs.hi[j], p.freqs.lo[j]);
    }
    named_bar_sync(3, 128);
    const float* drow = reinterpret_cast<const float*>(smem + L::off_dtab + (rb_i & 15) * L::DPITCH);
    const int i = rb_i;     // key row within the tile (rows >= BN idle)
    const int bb = i >> 4;  // block within the tile
    const bool row_in = i < BN;
    // Block start angles: this thread keeps the entries e = i + 128 k of the
    // table [NB][d/2] (all with pair jj = i % (d/2)) and advances them by the
    // angle BN * theta_jj per tile (a complex product), recomputing them
    // exactly every kAnchor tiles.
    constexpr int NE = (NB * HALF + 127) / 128;
    constexpr int kAnchor = 32;
    const int jj_own = i % HALF;
    const float2 rot = rope_cos_sin(BN, p.freqs.hi[jj_own], p.freqs.lo[jj_own]);
    float bc[NE], bs[NE];
    // Y arrives in quarters of 16 RoPE pairs from the Y issuer (warp 12):
    // quarter g of the loop in TMEM buffer g & 1, phase g >> 1 of
    // YFULL[g & 1]; each thread signals YFREE[g & 1] once it has the quarter
    // in registers. Every exit from this loop is decided by a barrier vote of
    // the whole warpgroup (bar.red.or), so no warp is left waiting at a named
    // barrier; a warp whose wait failed skips its work until the next vote.
    bool failed = false;
    for (int j = 0; j < U; ++j) {
      const int s = j % NST;
      // the previous tile's readers of btab are done past this barrier
      if (named_bar_or(3, 128, failed || *abort_flag != 0)) break;
      if (rebuild) {  // block start angles of this tile
#pragma unroll
        for (int k = 0; k < NE; ++k) {
          if (i + 128 * k >= NB * HALF) break;
          if (j % kAnchor == 0) {
            const float2 cs = rope_cos_sin_fast(j * BN + kBlock * ((i + 128 * k) / HALF), p.freqs.hi[jj_own],
                                                p.freqs.lo[jj_own]);
            bc[k] = cs.x;
            bs[k] = cs.y;
          } else {
            const float c = bc[k] * rot.x - bs[k] * rot.y;
            bs[k] = bs[k] * rot.x + bc[k] * rot.y;
            bc[k] = c;
          }
          btab[i + 128 * k] = make_float2(bc[k], bs[k]);
        }
      }
      failed = !wait_phase(bar(B_FULL + s), (j / NST) & 1, p.status);
      if (named_bar_or(3, 128, failed)) {  // also publishes btab to the warpgroup
        *abort_flag = 1;
        break;
      }
      const int mask = stage_mask[s];
      const int t = j * BN + i;
      const bool key_ok = row_in && ((mask >> bb) & 1) && t < Ls;
      uint8_t* kbuf = smem + s * L::STAGE + L::off_k;  // this tile's K buffer
      if (CODEC) {
        // Expand the tile's codes in place. Keys: each quarter-warp reads one
        // row's code bytes (contiguous: no bank conflicts), warp w the rows
        // 32 w ..; values: each thread its own row's three bit planes and norm.
        // Every code is read before any expanded row is written over them.
        constexpr int PR = D / 16, RPI = 32 / PR, NP = 32 / RPI;
        const int pc = lane % PR;
        uint4 kc[NP];
        float ksc[NP];
#pragma unroll
        for (int n = 0; n < NP; ++n) {
          const int row = 32 * (warp & 3) + RPI * n + lane / PR;
          kc[n] = make_uint4(0u, 0u, 0u, 0u);
          ksc[n] = 0.f;
          if (row < BN) {
            const uint8_t* kb = kbuf + (row >> 4) * codec_k_bytes(D);
            kc[n] = *reinterpret_cast<const uint4*>(kb + (row & 15) * D + 16 * pc);
            ksc[n] = __half2float(reinterpret_cast<const __half*>(kb + 16 * D)[(row & 15) * (D / 32) + pc / 2]);
          }
        }
        uint8_t* vbuf = smem + s * L::STAGE + L::off_v;
        uint32_t pw[3][D / 32];
        float nv = 0.f;
#pragma unroll
        for (int b = 0; b < 3; ++b)
#pragma unroll
          for (int gg = 0; gg < D / 32; ++gg) pw[b][gg] = 0u;
        if (row_in) {
          const uint8_t* vrow = vbuf + bb * codec_v_bytes(D);
#pragma unroll
          for (int b = 0; b < 3; ++b) {
            const uint8_t* pp = vrow + (i & 15) * (3 * D / 8) + b * (D / 8);
            if constexpr (D == 128) {
              const uint4 x = *reinterpret_cast<const uint4*>(pp);
              pw[b][0] = x.x;
              pw[b][1] = x.y;
              pw[b][2] = x.z;
              pw[b][3] = x.w;
            } else {
              const uint2 x = *reinterpret_cast<const uint2*>(pp);
              pw[b][0] = x.x;
              pw[b][1] = x.y;
            }
          }
          nv = *reinterpret_cast<const float*>(vrow + 6 * D + 4 * (i & 15));
        }
        named_bar_sync(3, 128);
        // K^ = q s, fp16; the pieces of the second 64-dim half store their
        // 16-byte halves in the other order (8 bank groups per quarter-warp)
#pragma unroll
        for (int n = 0; n < NP; ++n) {
          const int row = 32 * (warp & 3) + RPI * n + lane / PR;
          if (row < BN) {
            const uint32_t w[4] = {kc[n].x, kc[n].y, kc[n].z, kc[n].w};
            uint32_t o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint32_t x = w[e >> 1] >> (16 * (e & 1));
              o[e] = pack_f16(static_cast<float>(static_cast<int8_t>(x & 0xffu)) * ksc[n],
                              static_cast<float>(static_cast<int8_t>((x >> 8) & 0xffu)) * ksc[n]);
            }
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
              const int hf = hp ^ ((pc >> 2) & 1);
              const int dim = 16 * pc + 8 * hf;
              *reinterpret_cast<uint4*>(kbuf + (dim / 64) * (BN * 128) + swz<128>(row, (dim % 64) * 2)) =
                  hf ? make_uint4(o[4], o[5], o[6], o[7]) : make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
        }
        // V^ of this row in the rotated domain: c[code] ||v|| / sqrt(d) as bf16
        // (0 for keys outside the sequence or an unloaded block), by a
        // byte-permute table of the 8 scaled centroids
        if (row_in) {
          const float vs = key_ok ? nv * (1.0f / kSqrtD<D>) : 0.f;
          const uint32_t t0 = pack_bf16(p.vcent[0] * vs, p.vcent[1] * vs), t1 = pack_bf16(p.vcent[2] * vs, p.vcent[3] * vs);
          const uint32_t t2 = pack_bf16(p.vcent[4] * vs, p.vcent[5] * vs), t3 = pack_bf16(p.vcent[6] * vs, p.vcent[7] * vs);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {
            uint32_t o[4];
#pragma unroll
            for (int h4 = 0; h4 < 2; ++h4) {
              const int jd = 8 * c + 4 * h4, gw = jd >> 5, sh = jd & 31;
              const uint32_t lo2 = spread4((pw[0][gw] >> sh) & 15u) | (spread4((pw[1][gw] >> sh) & 15u) << 1);
              const uint32_t hi8 = spread4((pw[2][gw] >> sh) & 15u) * 0xffu;
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const uint32_t sel = 0x1010u + 0x22u * ((lo2 >> (16 * e)) & 0xffffu);
                const uint32_t m = __byte_perm(hi8, 0u, e ? 0x3322u : 0x1100u);
                o[2 * h4 + e] = (__byte_perm(t0, t1, sel) & ~m) | (__byte_perm(t2, t3, sel) & m);
              }
            }
            *reinterpret_cast<uint4*>(vbuf + (c / 8) * (BN * 128) + swz<128>(i, (c % 8) * 16)) =
                make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
      if (rebuild) {
        const float2* bt = btab + bb * HALF;
        // Rotates quarter q (pairs 16 q .. 16 q + 15: y[0..15] low dims, y[16..31]
        // their partners), adds K_base and writes fp16 K_a in place.
        auto rotate_quarter = [&](int q, const uint32_t (&y)[32]) {
          if (!key_ok) return;
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {  // 8 pairs per 16-byte chunk
            const int dlo = 16 * q + 8 * hc, dhi = dlo + HALF;
            // this thread's own K row: plain shared accesses the compiler may schedule
            uint4* plo = reinterpret_cast<uint4*>(kbuf + (dlo / 64) * (BN * 128) + swz<128>(i, (dlo % 64) * 2));
            uint4* phi = reinterpret_cast<uint4*>(kbuf + (dhi / 64) * (BN * 128) + swz<128>(i, (dhi % 64) * 2));
            const uint4 klo = *plo, khi = *phi;
            const uint32_t kl[4] = {klo.x, klo.y, klo.z, klo.w};
            const uint32_t kh[4] = {khi.x, khi.y, khi.z, khi.w};
            uint32_t olo[4], ohi[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              float rl[2], rh[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int pp = 8 * hc + 2 * w + e;  // pair index within the quarter
                const int jj = 16 * q + pp;
                const float2 b2 = bt[jj];
                const float cd = drow[2 * jj], sd = drow[2 * jj + 1];
                const float c = b2.x * cd - b2.y * sd;
                const float sn = b2.y * cd + b2.x * sd;
                const float yl = __uint_as_float(y[pp]), yh = __uint_as_float(y[16 + pp]);
                // K_base as loaded (bf16), or K^ expanded above (fp16)
                const float bl = CODEC ? (e ? f16_hi(kl[w]) : f16_lo(kl[w])) : (e ? bf16_hi(kl[w]) : bf16_lo(kl[w]));
                const float bh = CODEC ? (e ? f16_hi(kh[w]) : f16_lo(kh[w])) : (e ? bf16_hi(kh[w]) : bf16_lo(kh[w]));
                rl[e] = fmaf(yl, c, fmaf(-yh, sn, bl));
                rh[e] = fmaf(yh, c, fmaf(yl, sn, bh));
              }
              olo[w] = pack_f16(rl[0], rl[1]);
              ohi[w] = pack_f16(rh[0], rh[1]);
            }
            *plo = make_uint4(olo[0], olo[1], olo[2], olo[3]);
            *phi = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
          }
        };
        // Waits for quarter g and starts reading it from TMEM into y (the read
        // completes at the next tcgen05.wait::ld); false once a wait has failed.
        auto fetch_quarter = [&](int g, uint32_t (&y)[32]) -> bool {
          bool oky = !failed && wait_phase(bar(B_YFULL + (g & 1)), (g >> 1) & 1, p.status);
          oky = __all_sync(0xffffffffu, oky);
          if (!oky && !failed) {
            failed = true;
            *abort_flag = 1;
          }
          if (failed) return false;
          tc::fence_after();
          tc::ld_x32(tbase + lane_off + Y_COL + 32 * (g & 1), y);  // 16 low dims, then their partners
          return true;
        };
        // Quarters in pairs: while quarter q is rotated, quarter q + 1 is
        // already on its way out of TMEM (its own buffer, Y ping-pong).
        uint32_t ya[32], yb[32];
        const int g0 = j * NQ;
        bool have = fetch_quarter(g0, ya);
#pragma unroll 1
        for (int q = 0; q < NQ; q += 2) {
          const int g = g0 + q;
          if (!have) break;
          tc::wait_ld();
          tc::fence_before();
          mbar_arrive(bar(B_YFREE + (g & 1)));  // the buffer may take quarter g + 2
          const bool have_b = fetch_quarter(g + 1, yb);
          rotate_quarter(q, ya);
          if (!have_b) break;
          tc::wait_ld();
          tc::fence_before();
          mbar_arrive(bar(B_YFREE + ((g + 1) & 1)));
          have = q + 2 < NQ && fetch_quarter(g + 2, ya);
          rotate_quarter(q + 1, yb);
        }
      }
      if (failed) continue;
      // Keys past the sequence end or in a block that was not loaded: zero their
      // V and L_V rows, so that P = 0 there cannot meet stale (NaN) data.
      if (row_in && !key_ok) {
        uint8_t* vbuf = smem + s * L::STAGE + L::off_v;
        uint8_t* lvbuf = smem + s * L::STAGE + L::off_lv;
#pragma unroll
        for (int c = 0; c < (CODEC ? 0 : D / 8); ++c)  // a compressed tile's expansion wrote zeros already
          *reinterpret_cast<uint4*>(vbuf + (c / 8) * (BN * 128) + swz<128>(i, (c % 8) * 16)) = make_uint4(0, 0, 0, 0);
        if (use_lr) {
#pragma unroll
          for (int c = 0; c < LSPAN / 16; ++c)
            *reinterpret_cast<uint4*>(lvbuf + swz<LSPAN>(i, c * 16)) = make_uint4(0, 0, 0, 0);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      mbar_arrive(bar(B_KA + s));
    }
  }
  // ============================================================ Y issuer
  // Quarter g = L_K(tile g / NQ) B_K^T[rows 32 (g % NQ) ..] into Y buffer
  // g & 1, once the tile has landed and every rebuild thread has read
  // quarter g - 2 from that buffer.
  else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kLowRegs));
    if (warp == kYWarp && rebuild) {
      bool ok = true;
      for (int g = 0; g < NQ * U; ++g) {
        const int jj = g / NQ, q = g % NQ;
        if (uni(*abort_flag != 0) ||
            (g >= 2 && !uni(wait_phase(bar(B_YFREE + (g & 1)), ((g - 2) >> 1) & 1, p.status))) ||
            (q == 0 && !uni(wait_phase(bar(B_FULL + jj % NST), (jj / NST) & 1, p.status)))) {
          ok = false;
          break;
        }
        tc::fence_after();
        const uint32_t stj = sbase + (jj % NST) * L::STAGE;
        if (tc::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < RP / 16; ++kk) {
            const uint64_t a = tc::sdesc(stj + L::off_lk + kk * 32, 16, 8 * LSPAN, SW_LK);
            const uint64_t b = tc::sdesc(sbase + L::off_bk + 32 * q * LSPAN + kk * 32, 16, 8 * LSPAN, SW_LK);
            tc::mma_ss(tbase + Y_COL + 32 * (g & 1), a, b, kIdY, kk > 0);
          }
          tc::commit(bar(B_YFULL + (g & 1)));
        }
        __syncwarp();
      }
      if (!ok && lane == 0) *abort_flag = 1;
      if (uni(*abort_flag != 0)) {
        if (tc::elect_one()) {
          tc::commit(bar(B_DRAIN + 0));
          mbar_wait(bar(B_DRAIN + 0), 0, nullptr, 1u << 16);
        }
        __syncwarp();
      }
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
  p.lr_groups = cfg.lr_groups;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  rope_freqs(cfg, &p.freqs);
  const bool codec = cfg.kv_codec == LRKV_CODEC_POLYKV;
  p.cbase = static_cast<const uint8_t*>(a.base_pool);
  for (int k = 0; k < 8; ++k) p.vcent[k] = polykv_codec().centroid[k];
  CUtensorMap tb{}, tlk{}, tbr{}, tlr{};
  // a compressed base pool is read with plain bulk copies, block by block (no tensor maps)
  if (!codec && !make_pool_maps(cfg, a.base_pool, a.lr_pool, a.num_blocks, &tb, nullptr)) return LRKV_ERR_CUDA;
  if (!make_lr_map(cfg, a.lr_pool, a.num_blocks, PL<D, R>::RP, &tlk)) return LRKV_ERR_CUDA;
  if (!codec && !make_run_maps(cfg, a.base_pool, a.lr_pool, a.num_blocks, PL<D, R>::NB, PL<D, R>::RP, &tbr, &tlr))
    return LRKV_ERR_CUDA;
  auto kern = codec ? prefill_kernel<D, R, true> : prefill_kernel<D, R, false>;
  constexpr int smem = PL<D, R>::total;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), smem)) return LRKV_ERR_CUDA;
  const int tiles = (a.max_q_len * p.g + BM - 1) / BM;
  dim3 grid(tiles, cfg.n_kv_heads, a.num_seqs);
  kern<<<grid, kThreads, smem, stream>>>(p, tb, tlk, tbr, tlr);
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
