// Decode attention over the paged base + shared-A low-rank cache (bf16), on
// the 5th-generation tensor cores.
//
// LRAgent (arXiv 2602.01053), Abstract: one cached context serves every agent;
// each agent's adapter contribution is rebuilt from the low-rank cache at
// attention time, never expanded to full width in memory (Flash-LoRA-
// Attention). The V term is reordered as (P L_V) B_V and applied once, after
// the splits are merged.
//
// The K term. For a query row q (query n, head m, adapter a) and key token t
// with low-rank entry l(t) = L_K[t] (rank r), RoPE turns the pairs
// (j, j + d/2) by the angle t * theta_j, so the adapter part of the score is
//   q . RoPE_t(B_K,a^T l(t))
//     = sum_k l_k(t) sum_j [ cos(t theta_j) G_{k,j} + sin(t theta_j) G_{k,d/2+j} ]
//   G_{k,j}       = q_j B_{k,j} + q_{j+d/2} B_{k,j+d/2}
//   G_{k,d/2+j}   = q_{j+d/2} B_{k,j} - q_j B_{k,j+d/2}          (j < d/2)
// (the same sum as rotating the rebuilt row and taking the dot product, in
// another association order). G depends only on the query row and its
// adapter, so it is built once per work item; u(t) = [cos t theta, sin t theta]
// depends only on the position. Per 128-token tile the kernel then computes
//   W   = U G^T        (tokens x rows*r, tcgen05, fp16 operands)
//   S_b = K_base Q^T   (tokens x rows,   tcgen05, bf16)
//   s(t, row) = S_b(t, row) + sum_k l_k(t) W(t, row*r + k)     (one thread per token)
//   online softmax over tokens, P^T (bf16) to shared memory
//   O^T += V^T P^T,  O_lr^T += L_V^T P^T                        (tcgen05, bf16)
// so every agent's rows of one kv head share one pass over each base and
// low-rank tile, and the full-width adapter K is never formed.
//
// Work item: (context, chunk of <= 16 query rows of one kv head, split of the
// context's blocks, kv head), kv head fastest so that the items running
// together share the low-rank tiles through L2. One CTA per item:
//   warp 0      TMA producer: K_base + L_K tiles and V_base + L_V tiles of 8
//               blocks (per-block 2-D copies) into two rings
//   warp 1      issues W = U G^T (U from tensor memory)
//   warp 2      issues S_b = K_base Q^T
//   warp 3      issues O^T += V^T P^T and O_lr^T += L_V^T P^T
//   warps 4-7   one thread per token of the tile: U for the next tile, scores,
//               online softmax (rescale decided by a block-wide vote), P^T,
//               and at the end the split partial (m, l, O, O_lr)
// combine_kernel (launched after it on the same stream) merges the splits and
// applies B_V.
#include <math_constants.h>

#include <algorithm>
#include <climits>

#include "lrkv_device.cuh"
#include "lrkv_internal.h"
#include "tcgen05.cuh"

namespace lrkv {
namespace {

constexpr int kThreads = 384;
constexpr int kBT = 128;                   // tokens per tile (tcgen05 M)
constexpr int kTileBlocks = kBT / kBlock;  // 8 blocks per tile
constexpr int kMaxRows = 16;               // query rows per item (tcgen05 N of S_b, O^T)
constexpr int kSmemLimit = 227 * 1024;
constexpr int kMinSmem = 120 * 1024;       // keeps one CTA (and one TMEM owner) per SM
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns
constexpr uint32_t W_COL = 0;     // [<=256] W = U G^T, fp32
constexpr uint32_t DT_COL = 256;  // [d]    e^{i delta theta_j} of this lane's token offset, fp32
constexpr uint32_t U_COL = 384;   // [d/2]  U (fp16 pairs), operand A of W
constexpr uint32_t S_COL = 448;   // [16]   S_b
constexpr uint32_t OT_COL = 464;  // [16]   O^T  (lane = head dim)
constexpr uint32_t OL_COL = 480;  // [16]   O_lr^T (lane = rank index)
constexpr float kRescaleLog2 = 8.f;         // lazy rescale threshold (log2 units)
constexpr long long kWaitCycles = 1ll << 31;  // ~1 s: a wait this long has failed
constexpr long long kTestWaitCycles = 1ll << 20;  // the test-only stalled wait gives up after ~0.5 ms

struct DecodeParams {
  const __nv_bfloat16* q;
  const int32_t* ctx_q_start;
  const int32_t* adapter_ids;
  const int32_t* block_tables;
  const int32_t* ctx_lens;
  const __nv_bfloat16* B_K;
  const __nv_bfloat16* B_V;  // only prefetched here (applied by the combine kernel)
  float* part_ml;  // [Nq*Hq][S][2] (m in log2 units, l)
  float* part_o;   // [Nq*Hq][S][D + R]
  int32_t* status;
  int64_t num_blocks;
  int max_blocks, max_ctx_len, n_adapters, num_queries, Hq, Hkv, g;
  int lr_groups;  // > 1: agent-specific A, adapter a's low-rank group at columns [a r, (a+1) r)
  int test_stall;  // test only: the W issuer's first wait is on a barrier nobody arrives at
  int codec;       // compressed base pool (rebuild-mode kernel only): chunks of codec_chunk_bytes(D)
  const uint8_t* cbase;  // the compressed base pool
  float vcent[8];  // value-code centroids (Lloyd-Max for N(0,1)), ascending
  int rpi, n_chunks, n_splits, split_blocks;
  int has_bk, has_bv;
  float scale_log2;
  RopeFreqs freqs;
};

// Shared-memory layout (byte offsets from a 1024-aligned base), fixed per (d, r).
// One ring of NS slots carries the tiles in the order K_0, V_0, K_1, V_1, ...
// A slot holds [low-rank 128 x RP][base atoms: 64 dims x 128 tokens, 128-byte
// swizzle]: K_base + L_K for a K item, V_base + L_V for a V item.
template <int D, int R>
struct DL {
  static constexpr int HALF = D / 2;
  static constexpr int RP = R < 16 ? 16 : R;  // low-rank tile columns (zero past R)
  static constexpr int LSPAN = RP * 2;        // bytes per low-rank row
  static constexpr uint32_t SW_LR = tc::swizzle_code(LSPAN);
  static constexpr int RPI = (256 / R) < kMaxRows ? 256 / R : kMaxRows;  // rows per item
  static constexpr int RH = RPI / 2;          // rows per token warpgroup
  static constexpr int NW_MAX = RPI * R;      // W columns (<= 256)
  static constexpr int KATOMS = D / 64;
  static constexpr int ATOM = kBT * 128;
  static constexpr int LR_TILE = kBT * LSPAN;
  static constexpr int STAGE = LR_TILE + KATOMS * ATOM;
  static constexpr int GAMMA_ATOM = NW_MAX * 128;
  static constexpr int GAMMA = KATOMS * GAMMA_ATOM;
  static constexpr int QB = KATOMS * kMaxRows * 128;
  static constexpr int PB = 2 * kMaxRows * 128;  // P^T [16 rows][128 tokens] bf16
  static constexpr int BTAB = 2 * HALF * 8;
  static constexpr int MISC = 1024;
  static constexpr int TAIL = GAMMA + QB + 2 * PB + BTAB + MISC + 512;
  static constexpr int NS_FIT = (kSmemLimit - 1024 - TAIL) / STAGE;
  static constexpr int NS = NS_FIT > 4 ? 4 : NS_FIT;
  static constexpr int off_ring = 0;
  static constexpr int off_g = NS * STAGE;
  static constexpr int off_q = off_g + GAMMA;
  static constexpr int off_p = off_q + QB;
  static constexpr int off_btab = off_p + 2 * PB;
  static constexpr int off_misc = off_btab + BTAB;
  static constexpr int off_bar = off_misc + MISC;
  static constexpr int used = off_bar + 512;
  static constexpr int total = used + 1024;  // + alignment slack
  static_assert(NS >= 3, "the ring needs three slots");
  static_assert(total <= kSmemLimit, "decode tile does not fit in shared memory");
  static_assert(NW_MAX <= 256 && NW_MAX % 64 == 0 && RH >= 2, "W split over two warpgroups");
  // The M = 128 operands V^T (d = 64) and L_V^T (r < 128) read whole 128-row
  // spans; the rows past the tile land in the following buffers (never past
  // the allocation) and only feed accumulator lanes that are never read.
  static_assert((NS - 1) * STAGE + LR_TILE + 2 * ATOM <= used, "V^T span");
  static_assert((NS - 1) * STAGE + 7 * 16 * LSPAN + (128 / RP - 1) * LR_TILE + 16 * LSPAN <= used,
                "L_V^T span");
};

enum : int {
  B_FULL = 0,    // [4] ring slot full (TMA bytes)
  B_EMPTY = 4,   // [4] ring slot consumed: 8 token warps + two MMA commits (S_b twice; O^T and O_lr^T)
  B_UF = 8,      // U of the next tile written (8 token warps)
  B_WF = 9,      // W complete (commit)
  B_SF = 10,     // S_b complete (commit)
  B_WR = 11,     // W and S_b read out (8 token warps)
  B_PF = 12,     // [2] P^T written, O rescaled (8 token warps)
  B_PR = 14,     // [2] O^T and O_lr^T MMAs of that P buffer complete (two commits)
  B_DRAIN = 16,  // [4] per MMA warp, on abort: its MMAs have completed
  B_TEST = 20,   // test only: a barrier nothing arrives at (a bounded wait that must run out)
  B_GK = 21,     // the item's B_K rows landed in the G rows (TMA bytes)
  B_COUNT = 22
};

__device__ __forceinline__ uint32_t bar_count(int i) {
  if (i >= B_EMPTY && i < B_EMPTY + 4) return 10;
  if (i == B_UF || i == B_WR || i == B_PF || i == B_PF + 1) return 8;
  if (i == B_PR || i == B_PR + 1) return 2;
  return 1;
}

// Named barrier over `count` threads that also ORs a predicate across them.
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

// Waits for an mbarrier phase; gives up (LRKV_ERR_TIMEOUT, false) after
// kWaitCycles, or early once another role has raised the CTA's abort flag.
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

// A wait bounded by `limit` cycles (used by the test-only stall): gives up
// with LRKV_ERR_TIMEOUT like wait_ab.
__device__ __forceinline__ bool wait_limited(uint32_t bar, uint32_t parity, int32_t* st, long long limit) {
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) {
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

__device__ __forceinline__ bool warp_all(bool x) { return __all_sync(0xffffffffu, x); }

// Ring positions of tile j's K and V items in the issue order
// K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}.
__device__ __forceinline__ int kidx(int j, int n) { (void)n; return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int vidx(int j, int n) { return j + 1 < n ? 2 * j + 2 : 2 * j + 1; }

template <int D, int R>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeParams p,
                  const __grid_constant__ CUtensorMap tm_base,
                  const __grid_constant__ CUtensorMap tm_lr,
                  const __grid_constant__ CUtensorMap tm_bk) {
  using L = DL<D, R>;
  constexpr int HALF = D / 2;
  constexpr int KS = D / 16;  // k-steps over the head dims (and over u)
  constexpr int LSPAN = L::LSPAN;
  constexpr int NS = L::NS;
  constexpr int RH = L::RH;
  constexpr int WCH = RH * R / 32;  // W chunks (32 columns) per token warpgroup

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + L::off_bar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::off_misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::off_misc + 4);
  int* kmask = reinterpret_cast<int*>(smem + L::off_misc + 16);     // [4] loaded blocks per slot
  int* row_ad = reinterpret_cast<int*>(smem + L::off_misc + 32);    // [16]
  float* red = reinterpret_cast<float*>(smem + L::off_misc + 128);  // [2 groups][4 warps][8]
  float2* btab = reinterpret_cast<float2*>(smem + L::off_btab);     // [2][HALF]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- the work item (uniform across the CTA)
  int64_t rest = blockIdx.x;
  const int head = static_cast<int>(rest % p.Hkv);
  rest /= p.Hkv;
  const int split = static_cast<int>(rest % p.n_splits);
  rest /= p.n_splits;
  const int chunk = static_cast<int>(rest % p.n_chunks);
  const int ctx = static_cast<int>(rest / p.n_chunks);
  const int kbeg = split * p.split_blocks;
  const int32_t* btrow = p.block_tables + static_cast<int64_t>(ctx) * p.max_blocks;
  // block ids of the first two tiles, fetched before the context length is known
  int id0 = INT_MIN, id1 = INT_MIN;
  if (warp == 0) {
    const int kb = kbeg + (lane & 7) + (lane >> 3) * kTileBlocks;
    const int x = (lane < 2 * kTileBlocks && kb < p.max_blocks && kb < kbeg + p.split_blocks) ? __ldg(btrow + kb) : INT_MIN;
    id0 = __shfl_sync(0xffffffffu, x, lane & 7);
    id1 = __shfl_sync(0xffffffffu, x, (lane & 7) + 8);
    if (lane >= kTileBlocks) id0 = id1 = INT_MIN;
  } else if (p.n_adapters * R <= 4096) {
    // every adapter's B_K rows of this kv head into L2 (the rows this item
    // needs are known only after two dependent loads), and its B_V rows for
    // the combine kernel
    for (int i = tid - 32; i < p.n_adapters * R * (D / 64); i += kThreads - 32) {
      const int64_t off = (static_cast<int64_t>(i / (D / 64)) * p.Hkv + head) * D + 64 * (i % (D / 64));
      if (p.has_bk) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p.B_K + off));
      if (p.B_V != nullptr) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p.B_V + off));
    }
  }
  const int qs = __ldg(p.ctx_q_start + ctx), qe = __ldg(p.ctx_q_start + ctx + 1);
  int len = __ldg(p.ctx_lens + ctx);
  if (qs < 0 || qe > p.num_queries || qs > qe) {  // this context's query range is broken: skipped
    if (tid == 0) report(p.status, LRKV_ERR_INDEX);
    return;
  }
  // more queries on this context than max_q_per_ctx promised: the rows past
  // the last chunk get no partial (the combine zeroes their output)
  if (tid == 0 && chunk == 0 && split == 0 && (qe - qs) * p.g > p.n_chunks * p.rpi)
    report(p.status, LRKV_ERR_INDEX);
  const int row0 = chunk * p.rpi;
  const int nrows = min(p.rpi, (qe - qs) * p.g - row0);
  if (nrows <= 0) return;
  // agent-specific A: the item's rows all belong to one query (the plan makes
  // them so); its low-rank tiles are that adapter's group of columns
  int lr_x = 0;
  if (p.lr_groups > 1) {
    const int a0 = __ldg(p.adapter_ids + qs + row0 / p.g);
    if (a0 >= 0 && a0 < p.lr_groups) lr_x = a0 * R;
  }
  if (len < 1 || len > p.max_ctx_len) {
    if (tid == 0) report(p.status, LRKV_ERR_INDEX);
    len = 0;
  }
  const int nblk = (len + kBlock - 1) / kBlock;
  const int kend = min(kbeg + p.split_blocks, nblk);
  const int ntiles = kend > kbeg ? (kend - kbeg + kTileBlocks - 1) / kTileBlocks : 0;
  auto rec_of = [&](int r) -> int64_t {
    const int gr = row0 + r;
    const int n = qs + gr / p.g, m = head * p.g + gr % p.g;
    return (static_cast<int64_t>(n) * p.Hq + m) * p.n_splits + split;
  };
  if (ntiles == 0) {
    // An empty split still leaves a neutral partial (m = -inf, l = 0, O = 0).
    for (int i = tid; i < nrows * (D + R); i += kThreads)
      p.part_o[rec_of(i / (D + R)) * (D + R) + i % (D + R)] = 0.f;
    if (tid < nrows) {
      p.part_ml[2 * rec_of(tid)] = -CUDART_INF_F;
      p.part_ml[2 * rec_of(tid) + 1] = 0.f;
    }
    return;
  }

  // token warpgroups: e^{i delta theta_j} of this lane's token offset delta,
  // for the warpgroup's rotation pairs, computed while the setup loads and the
  // tensor-memory allocation are in flight (stored to TMEM after the barrier)
  constexpr int QH = HALF / 32;  // 16-pair chunks per token warpgroup
  uint32_t dvr[QH][32];
  if (warp >= 4) {
    const int jb0 = ((warp - 4) >> 2) * (HALF / 2);
    const int dl = (warp & 3) * 32 + lane;
#pragma unroll
    for (int q4 = 0; q4 < QH; ++q4)
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 cs = rope_cos_sin_fast(dl, p.freqs.hi[jb0 + 16 * q4 + i], p.freqs.lo[jb0 + 16 * q4 + i]);
        dvr[q4][2 * i] = __float_as_uint(cs.x);
        dvr[q4][2 * i + 1] = __float_as_uint(cs.y);
      }
  }

  // warps 1-3: this item's adapter ids and Q rows, requested before the setup barrier
  constexpr int QCH = kMaxRows * (D / 8);
  constexpr int QIT = (QCH + 95) / 96;
  uint4 qv[QIT];
  int a_row = -2;
  if (warp >= 1 && warp < 4) {
    const int pt = tid - 32;  // 0..95
    if (pt < nrows) a_row = __ldg(p.adapter_ids + qs + (row0 + pt) / p.g);
#pragma unroll
    for (int u = 0; u < QIT; ++u) {
      const int i = pt + 96 * u;
      const int r = i / (D / 8), c = i % (D / 8);
      qv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (i < QCH && r < nrows) {
        const int gr = row0 + r;
        const __nv_bfloat16* src =
            p.q + (static_cast<int64_t>(qs + gr / p.g) * p.Hq + head * p.g + gr % p.g) * D + 8 * c;
        qv[u] = __ldg(reinterpret_cast<const uint4*>(src));
      }
    }
  }

  // ---- barriers, tensor memory
  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), bar_count(i));
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tc::alloc(smem_u32(tmem_slot), kTmemCols);
  if (tid == 0) {
    prefetch_tmap(&tm_base);
    prefetch_tmap(&tm_lr);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tmem_slot;

  // Warp 1 (lane = item row): each row's B_K rows of its adapter, R rows of
  // d dims, by TMA straight into that row's G rows [r R, r R + R), 128-byte
  // swizzle like G. G is then built in place from shared memory. A row with
  // no adapter (or an id the combine reports as bad) gets a zero G row.
  bool gk_issued = false;
  if (warp == 1 && p.has_bk) {
    const bool ld = lane < nrows && a_row >= 0 && a_row < p.n_adapters;
    const uint32_t m = __ballot_sync(0xffffffffu, ld);
    gk_issued = m != 0;
    if (gk_issued) {
      if (lane == 0) mbar_arrive_expect_tx(bar(B_GK), __popc(m) * (R * D * 2));
      __syncwarp();
      if (ld) {
#pragma unroll
        for (int c = 0; c < L::KATOMS; ++c)
          tma_load_3d(sbase + L::off_g + c * L::GAMMA_ATOM + lane * (R * 128), &tm_bk, 64 * c, head, a_row * R,
                      bar(B_GK));
      }
    }
  }

  // ============================================================ producer
  // Items in the order K_0, K_1, V_0, K_2, V_1, ...: each K tile is requested
  // a tile ahead of the V tile before it, so V tiles (consumed last) do not
  // hold a slot while the next K tile could be landing.
  if (warp == 0) {
    const uint32_t bytes_k = L::KATOMS * 2048 + (p.has_bk ? 16 * LSPAN : 0);
    const uint32_t bytes_v = L::KATOMS * 2048 + (p.has_bv ? 16 * LSPAN : 0);
    auto tile_ids = [&](int j) -> int {  // this lane's block id of tile j
      const int kb = kbeg + j * kTileBlocks + lane;
      return (lane < kTileBlocks && kb < kend) ? __ldg(btrow + kb) : INT_MIN;
    };
    int id_a = (kbeg + lane < kend) ? id0 : INT_MIN;                // tile of the next V item
    int id_b = (kbeg + kTileBlocks + lane < kend) ? id1 : INT_MIN;  // tile of the next K item
    int id_c = ntiles > 2 ? tile_ids(2) : INT_MIN;
    bool ok = true;
    int issued = 0;
    auto issue = [&](int idx, int kind, int id) -> bool {
      bool valid = id != INT_MIN;
      if (valid && (id < 0 || id >= p.num_blocks)) {
        report(p.status, LRKV_ERR_INDEX);
        valid = false;
      }
      const uint32_t vm = __ballot_sync(0xffffffffu, valid);
      const int s = idx % NS;
      if (idx >= NS && !warp_all(wait_ab(bar(B_EMPTY + s), ((idx / NS) - 1) & 1, p.status, abort_flag)))
        return false;
      const uint32_t dst = sbase + L::off_ring + s * L::STAGE;
      const uint32_t fb = bar(B_FULL + s);
      if (lane == 0) {
        if (kind == 0) kmask[s] = static_cast<int>(vm);  // published by the arrive (release)
        mbar_arrive_expect_tx(fb, __popc(vm) * (kind == 0 ? bytes_k : bytes_v));
      }
      __syncwarp();
      if (valid) {
        const int y = ((id * 2 + kind) * p.Hkv + head) * kBlock;
#pragma unroll
        for (int a = 0; a < L::KATOMS; ++a)
          tma_load_2d(dst + L::LR_TILE + a * L::ATOM + lane * 2048, &tm_base, 64 * a, y, fb);
        if (kind == 0 ? p.has_bk : p.has_bv)
          tma_load_2d(dst + lane * 16 * LSPAN, &tm_lr, lr_x, (id * 2 + kind) * kBlock, fb);
      }
      return true;
    };
    ok = issue(kidx(0, ntiles), 0, id_a);
    issued = ok ? 1 : 0;
    for (int j = 0; ok && j < ntiles; ++j) {
      if (j + 1 < ntiles) {
        ok = issue(kidx(j + 1, ntiles), 0, id_b);
        if (!ok) break;
        ++issued;
      }
      ok = issue(vidx(j, ntiles), 1, id_a);
      if (!ok) break;
      ++issued;
      id_a = id_b;
      id_b = id_c;
      id_c = j + 3 < ntiles ? tile_ids(j + 3) : INT_MIN;
    }
    if (!ok && lane == 0) *abort_flag = 1;
    // No copy may still be landing when the CTA leaves: wait for the last
    // item issued into each slot (items are issued in index order).
    for (int s = 0; s < NS; ++s) {
      const int last = issued - 1 - ((issued - 1 - s) % NS + NS) % NS;
      if (last >= 0 && last < issued) wait_ab(bar(B_FULL + s), (last / NS) & 1, p.status, nullptr);
    }
  } else {
    // ================================================ prologue (warps 1-11)
    // Row adapters and Q (bf16, K-major, 128-byte swizzle; zero past nrows)
    // by warps 1-3; the token warpgroups meanwhile fill their rotation tables.
    const int gq = (warp - 4) >> 2;  // token warpgroup (warps 4-7: 0, 8-11: 1)
    const int tt = (warp & 3) * 32 + lane;  // token row of the tile = TMEM lane
    const uint32_t tl = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const int jb = gq * (HALF / 2);  // this warpgroup's rotation pairs [jb, jb + HALF/2)
    float th_hi = 0.f, th_lo = 0.f;
    if (warp >= 4 && tt < HALF / 2) {
      th_hi = p.freqs.hi[jb + tt];
      th_lo = p.freqs.lo[jb + tt];
    }
    if (warp < 4) {
      const int pt = tid - 32;  // 0..95
      if (pt < kMaxRows) {
        int a = a_row;
        if (pt < nrows && (a < -1 || a >= p.n_adapters || !p.has_bk)) a = -1;  // bad ids: reported by the combine
        row_ad[pt] = a;
      }
#pragma unroll
      for (int u = 0; u < QIT; ++u) {
        const int i = pt + 96 * u;
        const int r = i / (D / 8), c = i % (D / 8);
        if (i < QCH)
          *reinterpret_cast<uint4*>(smem + L::off_q + (c >> 3) * (kMaxRows * 128) + r * 128 +
                                    (((c & 7) ^ (r & 7)) << 4)) = qv[u];
      }
    } else {
      // the rotation table into TMEM (column 2j: cos, 2j + 1: sin)
#pragma unroll
      for (int q4 = 0; q4 < QH; ++q4) tc::st_x32(tl + DT_COL + 2 * (jb + 16 * q4), dvr[q4]);
      tc::wait_st();
      // base angles e^{i t0 theta_j} of tiles 0 and 1 (this warpgroup's pairs)
      const int t00 = kbeg * kBlock;
      if (tt < HALF / 2) {
        btab[jb + tt] = rope_cos_sin_fast(t00, th_hi, th_lo);
        if (ntiles > 1) btab[HALF + jb + tt] = rope_cos_sin_fast(t00 + kBT, th_hi, th_lo);
      }
    }
    named_bar_sync(1, kThreads - 32);
    bool use_w = false;
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) use_w |= row_ad[r] >= 0;
    const int nw = ((nrows * R + 15) / 16) * 16;

    // G (fp16, K-major over u, 128-byte swizzle) for rows n = row * R + k < nw,
    // one row per thread, in place over the B_K row that the TMA left there:
    // chunk pair (jc, d/16 + jc) of the row becomes (G_c, G_s) of the same pair.
    if (use_w) {
      const int n = tid - 32;
      if (n < nw) {
        const int r = n / R;
        uint8_t* grow = smem + L::off_g + n * 128;
        bool have = row_ad[r] >= 0;
        if (have && !wait_ab(bar(B_GK), 0, p.status, abort_flag)) {
          *abort_flag = 1;
          have = false;
        }
        const uint8_t* qrow = smem + L::off_q + r * 128;
#pragma unroll 2
        for (int jc = 0; jc < HALF / 8; ++jc) {
          const int c2 = HALF / 8 + jc;
          uint4* pa = reinterpret_cast<uint4*>(grow + (jc >> 3) * L::GAMMA_ATOM + (((jc & 7) ^ (n & 7)) << 4));
          uint4* pb = reinterpret_cast<uint4*>(grow + (c2 >> 3) * L::GAMMA_ATOM + (((c2 & 7) ^ (n & 7)) << 4));
          if (!have) {
            *pa = make_uint4(0u, 0u, 0u, 0u);
            *pb = make_uint4(0u, 0u, 0u, 0u);
            continue;
          }
          const uint4 q1 = *reinterpret_cast<const uint4*>(qrow + (jc >> 3) * (kMaxRows * 128) + (((jc & 7) ^ (r & 7)) << 4));
          const uint4 q2 = *reinterpret_cast<const uint4*>(qrow + (c2 >> 3) * (kMaxRows * 128) + (((c2 & 7) ^ (r & 7)) << 4));
          const uint4 b1 = *pa, b2 = *pb;
          const uint32_t qa[4] = {q1.x, q1.y, q1.z, q1.w};
          const uint32_t qb[4] = {q2.x, q2.y, q2.z, q2.w};
          const uint32_t ba[4] = {b1.x, b1.y, b1.z, b1.w};
          const uint32_t bb[4] = {b2.x, b2.y, b2.z, b2.w};
          uint32_t gc[4], gs[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float q1l = bf16_lo(qa[e]), q1h = bf16_hi(qa[e]);
            const float q2l = bf16_lo(qb[e]), q2h = bf16_hi(qb[e]);
            const float b1l = bf16_lo(ba[e]), b1h = bf16_hi(ba[e]);
            const float b2l = bf16_lo(bb[e]), b2h = bf16_hi(bb[e]);
            gc[e] = pack_f16(fmaf(q1l, b1l, q2l * b2l), fmaf(q1h, b1h, q2h * b2h));
            gs[e] = pack_f16(fmaf(q2l, b1l, -(q1l * b2l)), fmaf(q2h, b1h, -(q1h * b2h)));
          }
          *pa = make_uint4(gc[0], gc[1], gc[2], gc[3]);
          *pb = make_uint4(gs[0], gs[1], gs[2], gs[3]);
        }
      }
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // Q, G -> MMA operands
    named_bar_sync(1, kThreads - 32);

    if (warp == 1) {
      // ================================================ W issuer
      // Iteration j issues W_j = U_j G^T once U_j is written and W_{j-1} read.
      const uint32_t idw = tc::idesc_f16(128, nw, false, false, false);
      const uint64_t gdesc = tc::sdesc(sbase + L::off_g, 16, 1024, 2);
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        if (p.test_stall && j == 0) {
          // test only: a wait that runs out, then the abort path of every role
          ok = warp_all(wait_limited(bar(B_TEST), 0, p.status, kTestWaitCycles));
          if (!ok) break;
        }
        if (!use_w) break;
        ok = warp_all(wait_ab(bar(B_UF), j & 1, p.status, abort_flag));
        if (ok && j > 0) ok = warp_all(wait_ab(bar(B_WR), (j - 1) & 1, p.status, abort_flag));
        if (!ok) break;
        tc::fence_after();
        if (tc::elect_one()) {
#pragma unroll
          for (int k = 0; k < KS; ++k)
            tc::mma_ts(tbase + W_COL, tbase + U_COL + 8 * k,
                       gdesc + (((k >> 2) * L::GAMMA_ATOM + (k & 3) * 32) >> 4), idw, k > 0 ? 1u : 0u);
          tc::commit(bar(B_WF));
        }
        __syncwarp();
        ++issued;
      }
      if (!ok) {
        if (lane == 0) *abort_flag = 1;
        if (issued > 0) {
          if (tc::elect_one()) tc::commit(bar(B_DRAIN + 1));
          __syncwarp();
          wait_ab(bar(B_DRAIN + 1), 0, p.status, nullptr);
        }
      }
    } else if (warp == 2) {
      // ===================================================== S_b issuer
      const uint32_t ids = tc::idesc_f16(128, kMaxRows, true, false, false);
      const uint64_t qdesc = tc::sdesc(sbase + L::off_q, 16, 1024, 2);
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int ki = kidx(j, ntiles), s = ki % NS;
        ok = warp_all(wait_ab(bar(B_FULL + s), (ki / NS) & 1, p.status, abort_flag));
        if (ok && j > 0) ok = warp_all(wait_ab(bar(B_WR), (j - 1) & 1, p.status, abort_flag));
        if (!ok) break;
        tc::fence_after();
        if (tc::elect_one()) {
          const uint64_t kdesc = tc::sdesc(sbase + L::off_ring + s * L::STAGE + L::LR_TILE, 16, 1024, 2);
#pragma unroll
          for (int k = 0; k < KS; ++k)
            tc::mma_ss(tbase + S_COL, kdesc + (((k >> 2) * L::ATOM + (k & 3) * 32) >> 4),
                       qdesc + (((k >> 2) * (kMaxRows * 128) + (k & 3) * 32) >> 4), ids, k > 0 ? 1u : 0u);
          tc::commit(bar(B_SF));
          tc::commit(bar(B_EMPTY + s));
          tc::commit(bar(B_EMPTY + s));  // the slot's second MMA arrival (K items have one reader)
        }
        __syncwarp();
        ++issued;
      }
      if (!ok) {
        if (lane == 0) *abort_flag = 1;
        if (issued > 0) {
          if (tc::elect_one()) tc::commit(bar(B_DRAIN + 2));
          __syncwarp();
          wait_ab(bar(B_DRAIN + 2), 0, p.status, nullptr);
        }
      }
    } else if (warp == 3) {
      // ================================= O^T issuer, O_lr^T issuer
      // Both products of tile j read P_j: O^T += V_base^T P^T, then
      // O_lr^T += L_V^T P^T; together they release the V slot and the P buffer.
      const uint32_t ido = tc::idesc_f16(128, kMaxRows, true, true, false);
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int vi = vidx(j, ntiles), v = vi % NS, b = j & 1;
        ok = warp_all(wait_ab(bar(B_FULL + v), (vi / NS) & 1, p.status, abort_flag));
        if (ok) ok = warp_all(wait_ab(bar(B_PF + b), (j >> 1) & 1, p.status, abort_flag));
        if (!ok) break;
        tc::fence_after();
        if (tc::elect_one()) {
          const uint32_t vst = sbase + L::off_ring + v * L::STAGE;
          // V^T: M = head dims (MN-major; 64-dim atoms ATOM bytes apart), K = tokens
          const uint64_t vdesc = tc::sdesc(vst + L::LR_TILE, L::ATOM, 1024, 2);
          const uint64_t pdesc = tc::sdesc(sbase + L::off_p + b * L::PB, 16, 1024, 2);
#pragma unroll
          for (int k = 0; k < kBT / 16; ++k)
            tc::mma_ss(tbase + OT_COL, vdesc + ((k * 16 * 128) >> 4),
                       pdesc + (((k >> 2) * (kMaxRows * 128) + (k & 3) * 32) >> 4), ido,
                       (j > 0 || k > 0) ? 1u : 0u);
          if (p.has_bv) {
            // L_V^T: M = rank (MN-major, swizzled by the row span), K = tokens
            const uint64_t lvdesc = tc::sdesc(vst, L::LR_TILE, 8 * LSPAN, L::SW_LR);
#pragma unroll
            for (int k = 0; k < kBT / 16; ++k)
              tc::mma_ss(tbase + OL_COL, lvdesc + ((k * 16 * LSPAN) >> 4),
                         pdesc + (((k >> 2) * (kMaxRows * 128) + (k & 3) * 32) >> 4), ido,
                         (j > 0 || k > 0) ? 1u : 0u);
          }
          // two arrivals on each (the P buffer's and the V slot's MMA counts)
          tc::commit(bar(B_PR + b));
          tc::commit(bar(B_EMPTY + v));
          tc::commit(bar(B_PR + b));
          tc::commit(bar(B_EMPTY + v));
        }
        __syncwarp();
        ++issued;
      }
      if (!ok) {
        if (lane == 0) *abort_flag = 1;
        if (issued > 0) {
          if (tc::elect_one()) tc::commit(bar(B_DRAIN + 3));
          __syncwarp();
          wait_ab(bar(B_DRAIN + 3), 0, p.status, nullptr);
        }
      }
    } else {
      // ============================================ token warpgroups
      // Two warpgroups share the tile's 128 tokens (thread = token = TMEM
      // lane): warpgroup gq owns query rows [gq*RH, gq*RH + RH), their W
      // columns, their P^T rows and O columns, and rotation pairs [jb, jb + HALF/2).
      const int bar_g = 2 + gq;  // this warpgroup's named barrier
      const int rb = gq * RH;    // first row owned
      // U(t) = e^{i t0 theta} e^{i delta theta}, packed fp16 pairs:
      // columns [0, HALF/2) hold cos, [HALF/2, HALF) hold sin.
      auto build_u = [&](int bb) {
        const float2* bt = btab + bb * HALF;
#pragma unroll
        for (int q4 = 0; q4 < QH; ++q4) {
          const int j0 = jb + 16 * q4;
          uint32_t dv[32];
          tc::ld_x32(tl + DT_COL + 2 * j0, dv);
          tc::wait_ld();
          uint32_t uc[8], us[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 b2 = *reinterpret_cast<const float4*>(bt + j0 + 2 * i);
            const float cd0 = __uint_as_float(dv[4 * i]), sd0 = __uint_as_float(dv[4 * i + 1]);
            const float cd1 = __uint_as_float(dv[4 * i + 2]), sd1 = __uint_as_float(dv[4 * i + 3]);
            uc[i] = pack_f16(fmaf(b2.x, cd0, -(b2.y * sd0)), fmaf(b2.z, cd1, -(b2.w * sd1)));
            us[i] = pack_f16(fmaf(b2.y, cd0, b2.x * sd0), fmaf(b2.w, cd1, b2.z * sd1));
          }
          tc::st_x8(tl + U_COL + j0 / 2, uc);
          tc::st_x8(tl + U_COL + HALF / 2 + j0 / 2, us);
        }
        tc::wait_st();
      };
      if (use_w) {
        build_u(0);
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_UF));
      }

      float m_run[RH], l_run[RH];
#pragma unroll
      for (int r = 0; r < RH; ++r) {
        m_run[r] = -CUDART_INF_F;
        l_run[r] = 0.f;
      }
      // this warpgroup's W columns that exist: [gq*RH*R, min(nw, (gq+1)*RH*R))
      const int wch = use_w ? max(0, min(WCH, (nw - gq * RH * R + 31) / 32)) : 0;
      bool failed = false;
      for (int j = 0; j < ntiles; ++j) {
        const int ki = kidx(j, ntiles), vi = vidx(j, ntiles);
        const int s = ki % NS, v = vi % NS, b = j & 1;
        const int t0 = (kbeg + j * kTileBlocks) * kBlock;
        // ---- scores of this lane's token, own rows
        if (!failed && use_w) failed = !wait_ab(bar(B_WF), j & 1, p.status, abort_flag);
        if (!failed) failed = !wait_ab(bar(B_SF), j & 1, p.status, abort_flag);
        if (!failed) failed = !wait_ab(bar(B_FULL + s), (ki / NS) & 1, p.status, abort_flag);
        tc::fence_after();
        const int vmask = kmask[s];  // blocks of this tile that were loaded (valid ids inside the split)
        float sc[RH];
        {
          uint32_t sv[16];
          tc::ld_x16(tl + S_COL, sv);
          float slr[RH];
#pragma unroll
          for (int r = 0; r < RH; ++r) slr[r] = 0.f;
          if (wch > 0) {
            float lk[R];
            const uint8_t* lrow = smem + L::off_ring + s * L::STAGE;
#pragma unroll
            for (int c = 0; c < (R + 7) / 8; ++c) {
              const uint4 x = *reinterpret_cast<const uint4*>(lrow + swz<LSPAN>(tt, 16 * c));
              const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if (8 * c + 2 * e < R) lk[8 * c + 2 * e] = bf16_lo(xs[e]);
                if (8 * c + 2 * e + 1 < R) lk[8 * c + 2 * e + 1] = bf16_hi(xs[e]);
              }
            }
            // two chunks in flight per TMEM wait; two partial sums per row
            float acc2[RH];
#pragma unroll
            for (int r = 0; r < RH; ++r) acc2[r] = 0.f;
#pragma unroll
            for (int c = 0; c < WCH; c += 2) {
              if (c < wch) {
                uint32_t w0[32], w1[32];
                const uint32_t col = W_COL + gq * RH * R + 32 * c;
                tc::ld_x32(tl + col, w0);
                if (c + 1 < WCH) tc::ld_x32(tl + col + 32, w1);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  const int n = 32 * c + i;
                  slr[n / R] = fmaf(lk[n % R], __uint_as_float(w0[i]), slr[n / R]);
                }
                if (c + 1 < WCH && c + 1 < wch) {
#pragma unroll
                  for (int i = 0; i < 32; ++i) {
                    const int n = 32 * (c + 1) + i;
                    acc2[n / R] = fmaf(lk[n % R], __uint_as_float(w1[i]), acc2[n / R]);
                  }
                }
              }
            }
#pragma unroll
            for (int r = 0; r < RH; ++r) slr[r] += acc2[r];
          }
          tc::wait_ld();
#pragma unroll
          for (int r = 0; r < RH; ++r) sc[r] = __uint_as_float(gq ? sv[RH + r] : sv[r]) + slr[r];
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(B_WR));
          mbar_arrive(bar(B_EMPTY + s));
        }
        // ---- U of the next tile, base angles of the one after (own pairs)
        if (use_w && j + 1 < ntiles) {
          build_u((j + 1) & 1);
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_UF));
        }
        if (tt < HALF / 2 && j + 2 < ntiles) btab[b * HALF + jb + tt] = rope_cos_sin_fast(t0 + 2 * kBT, th_hi, th_lo);

        // ---- online softmax over the tile's tokens (log2 units), own rows.
        // Rows past the item's last row read W columns past nw, which hold
        // whatever an earlier kernel left in tensor memory: they are masked
        // here, so that they take no part in the rescale vote.
        const bool tok_ok = ((vmask >> (tt >> 4)) & 1) != 0 && t0 + tt < len;
        bool need = false;
#pragma unroll
        for (int r = 0; r < RH; ++r) {
          sc[r] = (tok_ok && rb + r < nrows) ? sc[r] * p.scale_log2 : -CUDART_INF_F;
          need |= sc[r] > m_run[r] + kRescaleLog2;
        }
        if (*abort_flag != 0) failed = true;
        if (named_bar_or(bar_g, 128, need || failed)) {  // also publishes btab
          if (named_bar_or(bar_g, 128, failed)) {
            failed = true;
            break;
          }
          float* rg = red + gq * 32;
#pragma unroll
          for (int r = 0; r < RH; ++r) {
            float x = sc[r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
            if (lane == 0) rg[(warp & 3) * 8 + r] = x;
          }
          named_bar_sync(bar_g, 128);
          float alpha[RH];
#pragma unroll
          for (int r = 0; r < RH; ++r) {
            const float mx = fmaxf(fmaxf(rg[r], rg[8 + r]), fmaxf(rg[16 + r], rg[24 + r]));
            const float mn = fmaxf(m_run[r], mx);
            alpha[r] = mn == -CUDART_INF_F ? 1.f : ex2(m_run[r] - mn);
            m_run[r] = mn;
            l_run[r] *= alpha[r];
          }
          named_bar_sync(bar_g, 128);  // rg is rewritten by the next vote's winners
          if (j > 0) {
            // the P V of the previous tile must have landed before O is rescaled
            if (!failed) failed = !wait_ab(bar(B_PR + ((j - 1) & 1)), ((j - 1) >> 1) & 1, p.status, abort_flag);
            tc::fence_after();
            uint32_t o[RH];
            tc::ld_cols<RH>(tl + OT_COL + rb, o);
            tc::wait_ld();
#pragma unroll
            for (int r = 0; r < RH; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
            tc::st_cols<RH>(tl + OT_COL + rb, o);
            if (p.has_bv) {
              tc::ld_cols<RH>(tl + OL_COL + rb, o);
              tc::wait_ld();
#pragma unroll
              for (int r = 0; r < RH; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
              tc::st_cols<RH>(tl + OL_COL + rb, o);
            }
            tc::wait_st();
          }
        }
#pragma unroll
        for (int r = 0; r < RH; ++r) {
          const float pr = ex2(sc[r] - (m_run[r] == -CUDART_INF_F ? 0.f : m_run[r]));
          l_run[r] += pr;
          sc[r] = pr;
        }
        // ---- P^T (bf16, K-major over tokens) once the P V two tiles back has read the buffer
        if (j >= 2 && !failed) failed = !wait_ab(bar(B_PR + b), ((j >> 1) - 1) & 1, p.status, abort_flag);
        {
          uint8_t* pb = smem + L::off_p + b * L::PB + (tt >> 6) * (kMaxRows * 128) + ((tt & 7) << 1);
          const int ch = (tt & 63) >> 3;
#pragma unroll
          for (int r = 0; r < RH; ++r)
            *reinterpret_cast<__nv_bfloat16*>(pb + (rb + r) * 128 + ((ch ^ ((rb + r) & 7)) << 4)) =
                __float2bfloat16_rn(sc[r]);
        }
        // rows of tokens outside the context or the split, or of blocks with a
        // bad id, hold stale memory: zero their V and L_V rows so that P = 0
        // there cannot meet a NaN (warpgroup 0: V atom 0, warpgroup 1: the rest)
        if (vmask != (1 << kTileBlocks) - 1 || t0 + kBT > len) {
          if (!failed) failed = !wait_ab(bar(B_FULL + v), (vi / NS) & 1, p.status, abort_flag);
          if (!tok_ok) {
            uint8_t* vst = smem + L::off_ring + v * L::STAGE;
            if (gq == 0) {
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(vst + L::LR_TILE + tt * 128 + 16 * c) = make_uint4(0u, 0u, 0u, 0u);
            } else {
#pragma unroll
              for (int a = 1; a < L::KATOMS; ++a)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                  *reinterpret_cast<uint4*>(vst + L::LR_TILE + a * L::ATOM + tt * 128 + 16 * c) =
                      make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
              for (int c = 0; c < LSPAN / 16; ++c)
                *reinterpret_cast<uint4*>(vst + tt * LSPAN + 16 * c) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        tc::fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(B_PF + b));
          mbar_arrive(bar(B_EMPTY + v));
        }
      }

      // ---- split partial: m, l, O, O_lr of each own row
      bool aborted = named_bar_or(bar_g, 128, failed);
      if (!aborted) {
        const bool okp = wait_ab(bar(B_PR + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, p.status, abort_flag);
        aborted = named_bar_or(bar_g, 128, !okp);
      }
      if (aborted) {
        if (tt == 0) *abort_flag = 1;
      } else {
        tc::fence_after();
        uint32_t o[RH], ol[RH];
        tc::ld_cols<RH>(tl + OT_COL + rb, o);
        tc::ld_cols<RH>(tl + OL_COL + rb, ol);
        tc::wait_ld();
        float* rg = red + gq * 32;
#pragma unroll
        for (int r = 0; r < RH; ++r) {
          float x = l_run[r];
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o2);
          if (lane == 0) rg[(warp & 3) * 8 + r] = x;
        }
        named_bar_sync(bar_g, 128);
#pragma unroll
        for (int r = 0; r < RH; ++r) {
          if (rb + r < nrows) {
            const int64_t rec = rec_of(rb + r);
            float* po = p.part_o + rec * (D + R);
            if (tt < D) po[tt] = __uint_as_float(o[r]);
            if (tt < R) po[D + tt] = p.has_bv ? __uint_as_float(ol[r]) : 0.f;
            if (tt == r) {
              p.part_ml[2 * rec] = m_run[r];
              p.part_ml[2 * rec + 1] = rg[r] + rg[8 + r] + rg[16 + r] + rg[24 + r];
            }
          }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    // no B_K copy may still be landing when the CTA leaves (an aborted item
    // may have skipped its wait)
    if (gk_issued && lane == 0) wait_ab(bar(B_GK), 0, p.status, nullptr);
    __syncwarp();
    tc::fence_after();
    tc::dealloc(tbase, kTmemCols);
  }
}

// ================================================================ rebuild mode
// Items whose rows all belong to one query, hence to one adapter (rank 64,
// four rows per item: a query's four heads of a kv head). The item keeps B_K^T
// of that adapter in shared memory (16 KB) instead of G (64 KB), and the
// adapter K term is rebuilt per tile on chip, as the pages describe it:
//   Y   = L_K B_K^T                      warp 1, tcgen05 (M = 128 tokens, N = d)
//   K_a = K_base + RoPE(Y)               token threads, fp16, in place of K_base
//   S   = K_a Q^T                        warp 2, tcgen05 (fp16)
//   O^T += V_base^T P^T, O_lr^T += L_V^T P^T   warps 3 and 1
// The two token warpgroups are two independent pipelines: warpgroup b takes
// the tiles j = b, b + 2, ... with its own Y, S, P, O and O_lr buffers and its
// own online softmax, and stores its own split partial (the combine merges
// 2 x n_splits partials per query head). While one warpgroup waits on a tensor
// or memory operation of its tile, the other works on the next tile.
namespace rb {
constexpr int kRows = 4;          // query rows per item (one query)
constexpr uint32_t RY_COL = 0;     // [2][d]  Y of the pipeline's tile, fp32
constexpr uint32_t RDT_COL = 256;  // [d]     e^{i delta theta_j} of this lane's token offset (cos, sin)
constexpr uint32_t RS_COL = 384;   // [2][16] S
constexpr uint32_t ROT_COL = 416;  // [2][16] O^T (lane = head dim)
constexpr uint32_t ROL_COL = 448;  // [2][16] O_lr^T (lane = rank index)

enum : int {
  FULL = 0,    // [4] ring slot full (TMA bytes)
  EMPTY = 4,   // [4] ring slot consumed: 4 token warps + two MMA commits
  YF = 8,      // [2] Y complete (commit)
  YR = 10,     // [2] Y read out (4 warps)
  KA = 12,     // [2] K_a written (4 warps)
  SF = 14,     // [2] S complete (commit)
  SR = 16,     // [2] S read out (4 warps)
  PF = 18,     // [2] P^T written, O rescaled (4 warps)
  PR = 20,     // [2] O^T and O_lr^T MMAs of that pipeline's tile complete (two commits)
  DRAIN = 22,  // [4] per MMA warp, on abort
  VX = 26,     // [2] compressed pool: V^ of that pipeline's tile expanded (4 warps)
  COUNT = 28
};

__device__ __forceinline__ uint32_t rb_bar_count(int i) {
  if (i >= EMPTY && i < EMPTY + 4) return 6;
  if ((i >= YR && i < YR + 2) || (i >= KA && i < KA + 2) || (i >= SR && i < SR + 2) || (i >= PF && i < PF + 2) ||
      (i >= VX && i < VX + 2))
    return 4;
  if (i >= PR && i < PR + 2) return 2;
  return 1;
}

// Shared-memory layout (byte offsets from a 1024-aligned base).
template <int D, int R>
struct Layout {
  static constexpr int HALF = D / 2;
  static constexpr int RP = R < 16 ? 16 : R;
  static constexpr int LSPAN = RP * 2;
  static constexpr uint32_t SW_LR = tc::swizzle_code(LSPAN);
  static constexpr int KATOMS = D / 64;
  static constexpr int ATOM = kBT * 128;
  static constexpr int LR_TILE = kBT * LSPAN;
  static constexpr int STAGE = LR_TILE + KATOMS * ATOM;
  static constexpr int BKT = D * LSPAN;  // B_K^T [d][r'] bf16, K-major, rows swizzled by LSPAN
  static constexpr int QB = KATOMS * kMaxRows * 128;
  static constexpr int PB = 2 * kMaxRows * 128;  // P^T [16 rows][128 tokens] bf16, per pipeline
  static constexpr int BTAB = 4 * HALF * 8;      // per pipeline, two buffers: base angles of its tiles
  static constexpr int MISC = 1024;
  static constexpr int TAIL = BKT + QB + 2 * PB + BTAB + MISC + 512;
  static constexpr int NS_FIT = (kSmemLimit - 1024 - TAIL) / STAGE;
  static constexpr int NS = NS_FIT > 4 ? 4 : NS_FIT;
  static constexpr int off_ring = 0;
  static constexpr int off_bk = NS * STAGE;
  static constexpr int off_q = off_bk + BKT;
  static constexpr int off_p = off_q + QB;
  static constexpr int off_btab = off_p + 2 * PB;
  static constexpr int off_misc = off_btab + BTAB;
  static constexpr int off_bar = off_misc + MISC;
  // the V^T operand of the last slot spans 128 head dims: at d = 64 the rows
  // past d (whose products are never read) may reach beyond the layout
  static constexpr int VSPAN = (NS - 1) * STAGE + LR_TILE + 2 * ATOM;
  static constexpr int used = off_bar + 512 > VSPAN ? off_bar + 512 : VSPAN;
  static constexpr int total = used + 1024;
  static_assert(NS >= 3, "the ring needs three slots");
  static_assert(total <= kSmemLimit, "decode tile does not fit in shared memory");
  static_assert(2 * D <= 256, "two Y buffers below the rotation table");
  static_assert((NS - 1) * STAGE + LR_TILE + 2 * ATOM <= used, "V^T span");
  static_assert((NS - 1) * STAGE + 7 * 16 * LSPAN + (128 / RP - 1) * LR_TILE + 16 * LSPAN <= used,
                "L_V^T span");
};
}  // namespace rb

template <int D, int R, bool CODEC>
__global__ void __launch_bounds__(kThreads, 1)
    decode_rb_kernel(const __grid_constant__ DecodeParams p,
                     const __grid_constant__ CUtensorMap tm_base,
                     const __grid_constant__ CUtensorMap tm_lr,
                     const __grid_constant__ CUtensorMap /* B_K map: G mode only */) {
  using L = rb::Layout<D, R>;
  using namespace rb;
  constexpr int HALF = D / 2;
  constexpr int KS = D / 16;
  constexpr int LSPAN = L::LSPAN;
  constexpr int NS = L::NS;
  constexpr int QH = HALF / 16;  // 16-pair chunks of a token's rotation

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + L::off_bar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::off_misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::off_misc + 4);
  int* kmask = reinterpret_cast<int*>(smem + L::off_misc + 16);     // [4] loaded blocks per slot
  float* red = reinterpret_cast<float*>(smem + L::off_misc + 128);  // [2 pipelines][4 warps][kRows]
  float2* btab = reinterpret_cast<float2*>(smem + L::off_btab);     // [2 pipelines][2][HALF]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- the work item (as in decode_kernel)
  int64_t rest = blockIdx.x;
  const int head = static_cast<int>(rest % p.Hkv);
  rest /= p.Hkv;
  const int split = static_cast<int>(rest % p.n_splits);
  rest /= p.n_splits;
  const int chunk = static_cast<int>(rest % p.n_chunks);
  const int ctx = static_cast<int>(rest / p.n_chunks);
  const int kbeg = split * p.split_blocks;
  const int32_t* btrow = p.block_tables + static_cast<int64_t>(ctx) * p.max_blocks;
  int id0 = INT_MIN, id1 = INT_MIN;
  if (warp == 0) {
    const int kb = kbeg + (lane & 7) + (lane >> 3) * kTileBlocks;
    const int x = (lane < 2 * kTileBlocks && kb < p.max_blocks && kb < kbeg + p.split_blocks) ? __ldg(btrow + kb) : INT_MIN;
    id0 = __shfl_sync(0xffffffffu, x, lane & 7);
    id1 = __shfl_sync(0xffffffffu, x, (lane & 7) + 8);
    if (lane >= kTileBlocks) id0 = id1 = INT_MIN;
  } else if (p.n_adapters * R <= 4096) {
    for (int i = tid - 32; i < p.n_adapters * R * (D / 64); i += kThreads - 32) {
      const int64_t off = (static_cast<int64_t>(i / (D / 64)) * p.Hkv + head) * D + 64 * (i % (D / 64));
      if (p.has_bk) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p.B_K + off));
      if (p.B_V != nullptr) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p.B_V + off));
    }
  }
  const int qs = __ldg(p.ctx_q_start + ctx), qe = __ldg(p.ctx_q_start + ctx + 1);
  int len = __ldg(p.ctx_lens + ctx);
  if (qs < 0 || qe > p.num_queries || qs > qe) {
    if (tid == 0) report(p.status, LRKV_ERR_INDEX);
    return;
  }
  if (tid == 0 && chunk == 0 && split == 0 && (qe - qs) * p.g > p.n_chunks * p.rpi)
    report(p.status, LRKV_ERR_INDEX);
  const int row0 = chunk * p.rpi;
  const int nrows = min(p.rpi, (qe - qs) * p.g - row0);
  if (nrows <= 0) return;
  // agent-specific A: the item's rows all belong to one query (the plan makes
  // them so); its low-rank tiles are that adapter's group of columns
  int lr_x = 0;
  if (p.lr_groups > 1) {
    const int a0 = __ldg(p.adapter_ids + qs + row0 / p.g);
    if (a0 >= 0 && a0 < p.lr_groups) lr_x = a0 * R;
  }
  if (len < 1 || len > p.max_ctx_len) {
    if (tid == 0) report(p.status, LRKV_ERR_INDEX);
    len = 0;
  }
  // the item's one adapter (a bad id scores as base only; the combine reports it)
  const int item_ad = __ldg(p.adapter_ids + qs + row0 / p.g);
  const bool rebuild = p.has_bk && item_ad >= 0 && item_ad < p.n_adapters;
  // compressed base pool: K tiles arrive as q8_0 codes and are expanded to
  // fp16 on chip (then scored in fp16 like a rebuilt K_a); V tiles arrive as
  // rotated 3-bit codes and are expanded to bf16 before the P V product
  constexpr bool codec = CODEC;  // a separate instantiation: the plain path carries none of it
  const bool kconv = rebuild || codec;
  const int nblk = (len + kBlock - 1) / kBlock;
  const int kend = min(kbeg + p.split_blocks, nblk);
  const int ntiles = kend > kbeg ? (kend - kbeg + kTileBlocks - 1) / kTileBlocks : 0;
  auto rec_of = [&](int r, int part) -> int64_t {
    const int gr = row0 + r;
    const int n = qs + gr / p.g, m = head * p.g + gr % p.g;
    return ((static_cast<int64_t>(n) * p.Hq + m) * p.n_splits + split) * 2 + part;
  };
  if (ntiles == 0) {
    for (int i = tid; i < 2 * nrows * (D + R); i += kThreads) {
      const int part = i / (nrows * (D + R)), k = i % (nrows * (D + R));
      p.part_o[rec_of(k / (D + R), part) * (D + R) + k % (D + R)] = 0.f;
    }
    if (tid < 2 * nrows) {
      p.part_ml[2 * rec_of(tid % nrows, tid / nrows)] = -CUDART_INF_F;
      p.part_ml[2 * rec_of(tid % nrows, tid / nrows) + 1] = 0.f;
    }
    return;
  }

  // token warps: e^{i delta theta_j} of this lane's token offset, for half of
  // the pairs (warpgroup b: pairs [b d/4, (b + 1) d/4)), stored after the barrier
  constexpr int QD = HALF / 32;
  uint32_t dvr[QD][32];
  if (warp >= 4) {
    const int jb0 = ((warp - 4) >> 2) * (HALF / 2);
    const int dl = (warp & 3) * 32 + lane;
#pragma unroll
    for (int q4 = 0; q4 < QD; ++q4)
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 cs = rope_cos_sin_fast(dl, p.freqs.hi[jb0 + 16 * q4 + i], p.freqs.lo[jb0 + 16 * q4 + i]);
        dvr[q4][2 * i] = __float_as_uint(cs.x);
        dvr[q4][2 * i + 1] = __float_as_uint(cs.y);
      }
  }
  // warps 1-3: Q rows of the item (fp16 when scored against fp16 K_a or K^)
  constexpr int QCH = kMaxRows * (D / 8);
  constexpr int QIT = (QCH + 95) / 96;
  uint4 qv[QIT];
  if (warp >= 1 && warp < 4) {
    const int pt = tid - 32;
#pragma unroll
    for (int u = 0; u < QIT; ++u) {
      const int i = pt + 96 * u;
      const int r = i / (D / 8), c = i % (D / 8);
      qv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (i < QCH && r < nrows) {
        const int gr = row0 + r;
        qv[u] = __ldg(reinterpret_cast<const uint4*>(
            p.q + (static_cast<int64_t>(qs + gr / p.g) * p.Hq + head * p.g + gr % p.g) * D + 8 * c));
      }
    }
  }

  // ---- barriers, tensor memory
  if (tid == 0) {
    for (int i = 0; i < COUNT; ++i) mbar_init(bar(i), rb_bar_count(i));
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tc::alloc(smem_u32(tmem_slot), kTmemCols);
  if (tid == 0) {
    if (!codec) prefetch_tmap(&tm_base);
    prefetch_tmap(&tm_lr);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ============================================================ producer
    // per block: K_base (or its codes Kq | Ks) and L_K; V_base (or Vq | Vn) and L_V
    const uint32_t kbase_bytes = codec ? codec_k_bytes(D) : L::KATOMS * 2048;
    const uint32_t vbase_bytes = codec ? codec_v_bytes(D) : L::KATOMS * 2048;
    const uint32_t bytes_k = kbase_bytes + (rebuild ? 16 * LSPAN : 0);
    const uint32_t bytes_v = vbase_bytes + (p.has_bv ? 16 * LSPAN : 0);
    auto tile_ids = [&](int j) -> int {
      const int kb = kbeg + j * kTileBlocks + lane;
      return (lane < kTileBlocks && kb < kend) ? __ldg(btrow + kb) : INT_MIN;
    };
    int id_a = (kbeg + lane < kend) ? id0 : INT_MIN;
    int id_b = (kbeg + kTileBlocks + lane < kend) ? id1 : INT_MIN;
    int id_c = ntiles > 2 ? tile_ids(2) : INT_MIN;
    bool ok = true;
    int issued = 0;
    auto issue = [&](int idx, int kind, int id) -> bool {
      bool valid = id != INT_MIN;
      if (valid && (id < 0 || id >= p.num_blocks)) {
        report(p.status, LRKV_ERR_INDEX);
        valid = false;
      }
      const uint32_t vm = __ballot_sync(0xffffffffu, valid);
      const int s = idx % NS;
      if (idx >= NS && !warp_all(wait_ab(bar(EMPTY + s), ((idx / NS) - 1) & 1, p.status, abort_flag)))
        return false;
      const uint32_t dst = sbase + L::off_ring + s * L::STAGE;
      const uint32_t fb = bar(FULL + s);
      if (lane == 0) {
        if (kind == 0) kmask[s] = static_cast<int>(vm);
        mbar_arrive_expect_tx(fb, __popc(vm) * (kind == 0 ? bytes_k : bytes_v));
      }
      __syncwarp();
      if (valid) {
        if (codec) {
          // the block's codes, staged at the front of the tile's K or V area
          const uint8_t* chunk = p.cbase + (static_cast<int64_t>(id) * p.Hkv + head) * codec_chunk_bytes(D);
          bulk_load(dst + L::LR_TILE + lane * (kind == 0 ? kbase_bytes : vbase_bytes),
                    chunk + (kind == 0 ? 0 : codec_k_bytes(D)), kind == 0 ? kbase_bytes : vbase_bytes, fb);
        } else {
          const int y = ((id * 2 + kind) * p.Hkv + head) * kBlock;
#pragma unroll
          for (int a = 0; a < L::KATOMS; ++a)
            tma_load_2d(dst + L::LR_TILE + a * L::ATOM + lane * 2048, &tm_base, 64 * a, y, fb);
        }
        if (kind == 0 ? rebuild : p.has_bv)
          tma_load_2d(dst + lane * 16 * LSPAN, &tm_lr, lr_x, (id * 2 + kind) * kBlock, fb);
      }
      return true;
    };
    ok = issue(kidx(0, ntiles), 0, id_a);
    issued = ok ? 1 : 0;
    for (int j = 0; ok && j < ntiles; ++j) {
      if (j + 1 < ntiles) {
        ok = issue(kidx(j + 1, ntiles), 0, id_b);
        if (!ok) break;
        ++issued;
      }
      ok = issue(vidx(j, ntiles), 1, id_a);
      if (!ok) break;
      ++issued;
      id_a = id_b;
      id_b = id_c;
      id_c = j + 3 < ntiles ? tile_ids(j + 3) : INT_MIN;
    }
    if (!ok && lane == 0) *abort_flag = 1;
    for (int s = 0; s < NS; ++s) {
      const int last = issued - 1 - ((issued - 1 - s) % NS + NS) % NS;
      if (last >= 0 && last < issued) wait_ab(bar(FULL + s), (last / NS) & 1, p.status, nullptr);
    }
  } else {
    // ================================================ prologue (warps 1-11)
    const int pb = (warp - 4) >> 2;  // token warps: pipeline (tiles pb, pb + 2, ...)
    const int tt = (warp & 3) * 32 + lane;
    const uint32_t tl = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    if (warp < 4) {
      const int pt = tid - 32;
#pragma unroll
      for (int u = 0; u < QIT; ++u) {
        const int i = pt + 96 * u;
        const int r = i / (D / 8), c = i % (D / 8);
        uint4 v = qv[u];
        if (kconv) {
          v.x = bf16x2_to_f16x2(v.x);
          v.y = bf16x2_to_f16x2(v.y);
          v.z = bf16x2_to_f16x2(v.z);
          v.w = bf16x2_to_f16x2(v.w);
        }
        if (i < QCH)
          *reinterpret_cast<uint4*>(smem + L::off_q + (c >> 3) * (kMaxRows * 128) + r * 128 +
                                    (((c & 7) ^ (r & 7)) << 4)) = v;
      }
      // B_K^T of the item's adapter: row n = head dim n, column k = rank index
      if (rebuild) {
        const __nv_bfloat16* src = p.B_K + static_cast<int64_t>(item_ad) * R * p.Hkv * D + head * D;
        for (int e = pt; e < D * (L::RP / 2); e += 96) {
          const int n = e % D, k0 = 2 * (e / D);
          const uint32_t lo = k0 < R ? __bfloat16_as_ushort(src[static_cast<int64_t>(k0) * p.Hkv * D + n]) : 0u;
          const uint32_t hi =
              k0 + 1 < R ? __bfloat16_as_ushort(src[static_cast<int64_t>(k0 + 1) * p.Hkv * D + n]) : 0u;
          *reinterpret_cast<uint32_t*>(smem + L::off_bk + swz<LSPAN>(n, 2 * k0)) = lo | (hi << 16);
        }
      }
    } else {
      const int jb = pb * (HALF / 2);
#pragma unroll
      for (int q4 = 0; q4 < QD; ++q4) tc::st_x32(tl + RDT_COL + 2 * (jb + 16 * q4), dvr[q4]);
      tc::wait_st();
      // base angles of the pipeline's first tile (tile pb)
      if (tt < HALF && pb < ntiles)
        btab[2 * pb * HALF + tt] = rope_cos_sin_fast((kbeg + pb * kTileBlocks) * kBlock, p.freqs.hi[tt], p.freqs.lo[tt]);
    }
    tc::fence_before();
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // Q, B_K^T -> MMA operands
    named_bar_sync(1, kThreads - 32);
    tc::fence_after();

    if (warp == 1) {
      // ======================================================== Y issuer
      const uint32_t idy = tc::idesc_f16(128, D, true, false, false);
      const uint64_t bdesc = tc::sdesc(sbase + L::off_bk, 16, 8 * LSPAN, L::SW_LR);
      bool ok = true;
      int issued = 0;
      for (int j = 0; rebuild && j < ntiles; ++j) {
        const int b = j & 1, i = j >> 1, ki = kidx(j, ntiles), s = ki % NS;
        ok = warp_all(wait_ab(bar(FULL + s), (ki / NS) & 1, p.status, abort_flag));
        if (ok && i > 0) ok = warp_all(wait_ab(bar(YR + b), (i - 1) & 1, p.status, abort_flag));
        if (!ok) break;
        tc::fence_after();
        if (tc::elect_one()) {
          const uint64_t ldesc = tc::sdesc(sbase + L::off_ring + s * L::STAGE, 16, 8 * LSPAN, L::SW_LR);
#pragma unroll
          for (int k = 0; k < L::RP / 16; ++k)
            tc::mma_ss(tbase + RY_COL + b * D, ldesc + 2 * k, bdesc + 2 * k, idy, k > 0 ? 1u : 0u);
          tc::commit(bar(YF + b));
        }
        __syncwarp();
        ++issued;
      }
      if (!ok) {
        if (lane == 0) *abort_flag = 1;
        if (issued > 0) {
          if (tc::elect_one()) tc::commit(bar(DRAIN + 1));
          __syncwarp();
          wait_ab(bar(DRAIN + 1), 0, p.status, nullptr);
        }
      }
    } else if (warp == 2) {
      // ======================================================== S issuer
      const uint32_t ids = tc::idesc_f16(128, kMaxRows, !kconv, false, false);
      const uint64_t qdesc = tc::sdesc(sbase + L::off_q, 16, 1024, 2);
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int b = j & 1, i = j >> 1, ki = kidx(j, ntiles), s = ki % NS;
        ok = warp_all(wait_ab(bar(FULL + s), (ki / NS) & 1, p.status, abort_flag));
        if (ok) ok = warp_all(wait_ab(bar(KA + b), i & 1, p.status, abort_flag));
        if (ok && i > 0) ok = warp_all(wait_ab(bar(SR + b), (i - 1) & 1, p.status, abort_flag));
        if (!ok) break;
        tc::fence_after();
        if (tc::elect_one()) {
          const uint64_t kdesc = tc::sdesc(sbase + L::off_ring + s * L::STAGE + L::LR_TILE, 16, 1024, 2);
#pragma unroll
          for (int k = 0; k < KS; ++k)
            tc::mma_ss(tbase + RS_COL + 16 * b, kdesc + (((k >> 2) * L::ATOM + (k & 3) * 32) >> 4),
                       qdesc + (((k >> 2) * (kMaxRows * 128) + (k & 3) * 32) >> 4), ids, k > 0 ? 1u : 0u);
          tc::commit(bar(SF + b));
          tc::commit(bar(EMPTY + s));
          tc::commit(bar(EMPTY + s));  // K items have one MMA reader after the rebuild: both arrivals here
        }
        __syncwarp();
        ++issued;
      }
      if (!ok) {
        if (lane == 0) *abort_flag = 1;
        if (issued > 0) {
          if (tc::elect_one()) tc::commit(bar(DRAIN + 2));
          __syncwarp();
          wait_ab(bar(DRAIN + 2), 0, p.status, nullptr);
        }
      }
    } else if (warp == 3) {
      // ================================= O^T issuer, O_lr^T issuer
      // Both products of a tile read its P: O^T += V^T P^T, then O_lr^T += L_V^T P^T.
      const uint32_t ido = tc::idesc_f16(128, kMaxRows, true, true, false);
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int b = j & 1, i = j >> 1, vi = vidx(j, ntiles), v = vi % NS;
        ok = warp_all(wait_ab(bar(FULL + v), (vi / NS) & 1, p.status, abort_flag));
        if (ok) ok = warp_all(wait_ab(bar(PF + b), i & 1, p.status, abort_flag));
        if (ok && codec) ok = warp_all(wait_ab(bar(VX + b), i & 1, p.status, abort_flag));
        if (!ok) break;
        tc::fence_after();
        if (tc::elect_one()) {
          const uint32_t vst = sbase + L::off_ring + v * L::STAGE;
          const uint64_t vdesc = tc::sdesc(vst + L::LR_TILE, L::ATOM, 1024, 2);
          const uint64_t pdesc = tc::sdesc(sbase + L::off_p + b * L::PB, 16, 1024, 2);
#pragma unroll
          for (int k = 0; k < kBT / 16; ++k)
            tc::mma_ss(tbase + ROT_COL + 16 * b, vdesc + ((k * 16 * 128) >> 4),
                       pdesc + (((k >> 2) * (kMaxRows * 128) + (k & 3) * 32) >> 4), ido,
                       (i > 0 || k > 0) ? 1u : 0u);
          if (p.has_bv) {
            const uint64_t lvdesc = tc::sdesc(vst, L::LR_TILE, 8 * LSPAN, L::SW_LR);
#pragma unroll
            for (int k = 0; k < kBT / 16; ++k)
              tc::mma_ss(tbase + ROL_COL + 16 * b, lvdesc + ((k * 16 * LSPAN) >> 4),
                         pdesc + (((k >> 2) * (kMaxRows * 128) + (k & 3) * 32) >> 4), ido,
                         (i > 0 || k > 0) ? 1u : 0u);
          }
          // two arrivals on each (the P buffer's and the V slot's MMA counts)
          tc::commit(bar(PR + b));
          tc::commit(bar(EMPTY + v));
          tc::commit(bar(PR + b));
          tc::commit(bar(EMPTY + v));
        }
        __syncwarp();
        ++issued;
      }
      if (!ok) {
        if (lane == 0) *abort_flag = 1;
        if (issued > 0) {
          if (tc::elect_one()) tc::commit(bar(DRAIN + 3));
          __syncwarp();
          wait_ab(bar(DRAIN + 3), 0, p.status, nullptr);
        }
      }
    } else {
      // ================================== token pipelines (warps 4-7, 8-11)
      const int bar_g = 2 + pb;
      // base angles: the i-th tile of this pipeline reads buffer i & 1; the
      // (i+1)-th tile's are written into the other buffer, which every thread
      // of the pipeline finished reading before the previous tile's vote
      float2* btp = btab + 2 * pb * HALF;
      float m_run[kRows], l_run[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        m_run[r] = -CUDART_INF_F;
        l_run[r] = 0.f;
      }
      const float th_hi = tt < HALF ? p.freqs.hi[tt] : 0.f, th_lo = tt < HALF ? p.freqs.lo[tt] : 0.f;
      bool failed = false;
      // Compressed pool: V^ of this pipeline's previous tile, in the rotated
      // domain, c[code_j] ||v|| / sqrt(d), bf16, expanded over the staged codes
      // once this pipeline reaches its next tile (the codes landed long ago):
      // every thread first takes its row's codes, then all write. Rows outside
      // the context, the split or a loaded block get 0. The combine rotates the
      // merged sum back.
      int prev_v = 0;
      uint32_t prev_vpar = 0;
      bool prev_tok = false, pending_v = false;
      auto expand_v = [&](int vs_slot, uint32_t vpar, bool ok_tok) {
        if (!failed) failed = !wait_ab(bar(FULL + vs_slot), vpar, p.status, abort_flag);
        uint8_t* vst = smem + L::off_ring + vs_slot * L::STAGE;
        uint8_t* vt = vst + L::LR_TILE;
        const uint8_t* vrow = vt + (tt >> 4) * codec_v_bytes(D);
        // each bit plane of the row in one load (rows 3 d / 8 bytes apart: no bank conflicts)
        uint32_t pw[3][D / 32];
#pragma unroll
        for (int b = 0; b < 3; ++b) {
          const uint8_t* pp = vrow + (tt & 15) * (3 * D / 8) + b * (D / 8);
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
        const float nv = *reinterpret_cast<const float*>(vrow + 6 * D + 4 * (tt & 15));
        named_bar_sync(bar_g, 128);
        const float vs = ok_tok ? nv * (1.0f / kSqrtD<D>) : 0.f;
        // the 8 scaled centroids as bf16: codes 0-3 in {t1:t0}, 4-7 in {t3:t2}
        const uint32_t t0 = pack_bf16(p.vcent[0] * vs, p.vcent[1] * vs), t1 = pack_bf16(p.vcent[2] * vs, p.vcent[3] * vs);
        const uint32_t t2 = pack_bf16(p.vcent[4] * vs, p.vcent[5] * vs), t3 = pack_bf16(p.vcent[6] * vs, p.vcent[7] * vs);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {  // dims 8c .. 8c + 7
          uint32_t o[4];
#pragma unroll
          for (int h4 = 0; h4 < 2; ++h4) {  // 4 dims: their code bits spread to one byte each
            const int j = 8 * c + 4 * h4, g = j >> 5, sh = j & 31;
            const uint32_t lo2 = spread4((pw[0][g] >> sh) & 15u) | (spread4((pw[1][g] >> sh) & 15u) << 1);
            const uint32_t hi8 = spread4((pw[2][g] >> sh) & 15u) * 0xffu;  // 0xff where code >= 4
#pragma unroll
            for (int e = 0; e < 2; ++e) {  // a pair of dims: byte selectors 2l, 2l + 1 per element
              const uint32_t sel = 0x1010u + 0x22u * ((lo2 >> (16 * e)) & 0xffffu);
              const uint32_t m = __byte_perm(hi8, 0u, e ? 0x3322u : 0x1100u);
              o[2 * h4 + e] = (__byte_perm(t0, t1, sel) & ~m) | (__byte_perm(t2, t3, sel) & m);
            }
          }
          *reinterpret_cast<uint4*>(vt + ((8 * c) >> 6) * L::ATOM + swz<128>(tt, ((8 * c) & 63) * 2)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // V^ -> P V operand
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(VX + pb));
          mbar_arrive(bar(EMPTY + vs_slot));
        }
        pending_v = false;
      };
      int i = 0;
      for (int j = pb; j < ntiles; j += 2, ++i) {
        const int ki = kidx(j, ntiles), vi = vidx(j, ntiles);
        const int s = ki % NS, v = vi % NS;
        const uint32_t ph = i & 1;
        const int t0 = (kbeg + j * kTileBlocks) * kBlock;
        if (pending_v) expand_v(prev_v, prev_vpar, prev_tok);
        // ---- K_a = K_base + RoPE(Y) for this lane's token, every pair, fp16 in place
        if (kconv) {
          if (!failed && rebuild) failed = !wait_ab(bar(YF + pb), ph, p.status, abort_flag);
          if (!failed) failed = !wait_ab(bar(FULL + s), (ki / NS) & 1, p.status, abort_flag);
          tc::fence_after();
          uint8_t* kt = smem + L::off_ring + s * L::STAGE + L::LR_TILE;
          if (codec) {
            // K^ = q s (q8_0), fp16, over the staged codes. Each quarter-warp
            // takes one row's D code bytes as 16-byte pieces (contiguous: no
            // bank conflicts), warp w the rows 32 (w % 4) ..; all the pipeline's
            // codes are read before any expanded row is written over them.
            constexpr int PR = D / 16;             // 16-byte pieces per row
            constexpr int RPI = 32 / PR;           // rows per warp pass
            constexpr int NP = 32 / RPI;           // passes over the warp's 32 rows
            const int pc = lane % PR;              // this thread's piece: dims 16 pc ..
            uint4 kc[NP];
            float ksc[NP];
#pragma unroll
            for (int i = 0; i < NP; ++i) {
              const int row = 32 * (warp & 3) + RPI * i + lane / PR;
              const uint8_t* kb = kt + (row >> 4) * codec_k_bytes(D);
              kc[i] = *reinterpret_cast<const uint4*>(kb + (row & 15) * D + 16 * pc);
              ksc[i] = __half2float(reinterpret_cast<const __half*>(kb + 16 * D)[(row & 15) * (D / 32) + pc / 2]);
            }
            named_bar_sync(bar_g, 128);
#pragma unroll
            for (int i = 0; i < NP; ++i) {
              const int row = 32 * (warp & 3) + RPI * i + lane / PR;
              const uint32_t w[4] = {kc[i].x, kc[i].y, kc[i].z, kc[i].w};
              uint32_t o[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const uint32_t x = w[e >> 1] >> (16 * (e & 1));
                o[e] = pack_f16(static_cast<float>(static_cast<int8_t>(x & 0xffu)) * ksc[i],
                                static_cast<float>(static_cast<int8_t>((x >> 8) & 0xffu)) * ksc[i]);
              }
              // the pieces of atom 1 store their halves in the other order, so
              // that the 8 stores of one row's quarter-warp hit 8 bank groups
#pragma unroll
              for (int hp = 0; hp < 2; ++hp) {
                const int hf = hp ^ ((pc >> 2) & 1);
                const int dim = 16 * pc + 8 * hf;
                *reinterpret_cast<uint4*>(kt + (dim >> 6) * L::ATOM + swz<128>(row, (dim & 63) * 2)) =
                    hf ? make_uint4(o[4], o[5], o[6], o[7]) : make_uint4(o[0], o[1], o[2], o[3]);
              }
            }
          }
          if (rebuild) {
          const uint32_t ycol = RY_COL + pb * D;
          const float2* bt = btp + (i & 1) * HALF;
#pragma unroll 1
          for (int q4 = 0; q4 < QH; ++q4) {
            const int j0 = 16 * q4;
            uint32_t dv[32], ylo[16], yhi[16];
            tc::ld_x32(tl + RDT_COL + 2 * j0, dv);
            tc::ld_x16(tl + ycol + j0, ylo);
            tc::ld_x16(tl + ycol + HALF + j0, yhi);
            tc::wait_ld();
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {  // 8 pairs per 16-byte chunk
              const int dlo = j0 + 8 * hc, dhi = dlo + HALF;
              uint4* plo = reinterpret_cast<uint4*>(kt + (dlo >> 6) * L::ATOM + swz<128>(tt, (dlo & 63) * 2));
              uint4* phi = reinterpret_cast<uint4*>(kt + (dhi >> 6) * L::ATOM + swz<128>(tt, (dhi & 63) * 2));
              const uint4 klo = *plo, khi = *phi;
              const uint32_t kl[4] = {klo.x, klo.y, klo.z, klo.w};
              const uint32_t kh[4] = {khi.x, khi.y, khi.z, khi.w};
              uint32_t olo[4], ohi[4];
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                float rl[2], rh[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int k = 8 * hc + 2 * w + e;  // pair j0 + k
                  const float2 b2 = bt[j0 + k];
                  const float cd = __uint_as_float(dv[2 * k]), sd = __uint_as_float(dv[2 * k + 1]);
                  const float c = fmaf(b2.x, cd, -(b2.y * sd)), sn = fmaf(b2.y, cd, b2.x * sd);
                  const float yl = __uint_as_float(ylo[k]), yh = __uint_as_float(yhi[k]);
                  // K_base as loaded (bf16), or K^ expanded above (fp16)
                  const float bl = codec ? (e ? f16_hi(kl[w]) : f16_lo(kl[w])) : (e ? bf16_hi(kl[w]) : bf16_lo(kl[w]));
                  const float bh = codec ? (e ? f16_hi(kh[w]) : f16_lo(kh[w])) : (e ? bf16_hi(kh[w]) : bf16_lo(kh[w]));
                  rl[e] = fmaf(yl, c, fmaf(-yh, sn, bl));
                  rh[e] = fmaf(yh, c, fmaf(yl, sn, bh));
                }
                olo[w] = pack_f16(rl[0], rl[1]);
                ohi[w] = pack_f16(rh[0], rh[1]);
              }
              *plo = make_uint4(olo[0], olo[1], olo[2], olo[3]);
              *phi = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
            }
          }
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(YR + pb));
          }
          asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // K_a or K^ -> S operand
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(KA + pb));

        // ---- scores of this lane's token, every row
        if (!failed) failed = !wait_ab(bar(SF + pb), ph, p.status, abort_flag);
        if (!failed) failed = !wait_ab(bar(FULL + s), (ki / NS) & 1, p.status, abort_flag);
        tc::fence_after();
        const int vmask = kmask[s];
        float sc[kRows];
        {
          uint32_t sv[kRows];
          tc::ld_cols<kRows>(tl + RS_COL + 16 * pb, sv);
          tc::wait_ld();
#pragma unroll
          for (int r = 0; r < kRows; ++r) sc[r] = __uint_as_float(sv[r]);
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(SR + pb));
          mbar_arrive(bar(EMPTY + s));
        }
        // base angles of this pipeline's next tile (j + 2), published by the vote below
        if (tt < HALF && j + 2 < ntiles) btp[((i + 1) & 1) * HALF + tt] = rope_cos_sin_fast(t0 + 2 * kBT, th_hi, th_lo);

        // ---- online softmax over the tile's tokens (log2 units)
        const bool tok_ok = ((vmask >> (tt >> 4)) & 1) != 0 && t0 + tt < len;
        bool need = false;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          sc[r] = tok_ok ? sc[r] * p.scale_log2 : -CUDART_INF_F;
          need |= sc[r] > m_run[r] + kRescaleLog2;
        }
        if (*abort_flag != 0) failed = true;
        if (named_bar_or(bar_g, 128, need || failed)) {  // also publishes bt
          if (named_bar_or(bar_g, 128, failed)) {
            failed = true;
            break;
          }
          float* rg = red + pb * 4 * kRows;
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            float x = sc[r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
            if (lane == 0) rg[(warp & 3) * kRows + r] = x;
          }
          named_bar_sync(bar_g, 128);
          float alpha[kRows];
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            const float mx = fmaxf(fmaxf(rg[r], rg[kRows + r]), fmaxf(rg[2 * kRows + r], rg[3 * kRows + r]));
            const float mn = fmaxf(m_run[r], mx);
            alpha[r] = mn == -CUDART_INF_F ? 1.f : ex2(m_run[r] - mn);
            m_run[r] = mn;
            l_run[r] *= alpha[r];
          }
          named_bar_sync(bar_g, 128);
          if (i > 0) {
            // the P V of this pipeline's previous tile must have landed before O is rescaled
            if (!failed) failed = !wait_ab(bar(PR + pb), (i - 1) & 1, p.status, abort_flag);
            tc::fence_after();
            uint32_t o[kRows];
            tc::ld_cols<kRows>(tl + ROT_COL + 16 * pb, o);
            tc::wait_ld();
#pragma unroll
            for (int r = 0; r < kRows; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
            tc::st_cols<kRows>(tl + ROT_COL + 16 * pb, o);
            if (p.has_bv) {
              tc::ld_cols<kRows>(tl + ROL_COL + 16 * pb, o);
              tc::wait_ld();
#pragma unroll
              for (int r = 0; r < kRows; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
              tc::st_cols<kRows>(tl + ROL_COL + 16 * pb, o);
            }
            tc::wait_st();
          }
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          const float pr = ex2(sc[r] - (m_run[r] == -CUDART_INF_F ? 0.f : m_run[r]));
          l_run[r] += pr;
          sc[r] = pr;
        }
        // ---- P^T (bf16, K-major over tokens) once this pipeline's previous P V has read it
        if (i > 0 && !failed) failed = !wait_ab(bar(PR + pb), (i - 1) & 1, p.status, abort_flag);
        {
          uint8_t* pbuf = smem + L::off_p + pb * L::PB + (tt >> 6) * (kMaxRows * 128) + ((tt & 7) << 1);
          const int ch = (tt & 63) >> 3;
#pragma unroll
          for (int r = 0; r < kRows; ++r)
            *reinterpret_cast<__nv_bfloat16*>(pbuf + r * 128 + ((ch ^ (r & 7)) << 4)) = __float2bfloat16_rn(sc[r]);
        }
        if (vmask != (1 << kTileBlocks) - 1 || t0 + kBT > len) {
          // V and L_V rows of tokens outside the context, the split or a loaded
          // block hold stale memory: zero them so that P = 0 cannot meet a NaN
          // (a compressed V tile still holds every row's codes: its expansion
          // zeroes those rows instead)
          if (!failed) failed = !wait_ab(bar(FULL + v), (vi / NS) & 1, p.status, abort_flag);
          if (!tok_ok) {
            uint8_t* vst = smem + L::off_ring + v * L::STAGE;
#pragma unroll
            for (int a = 0; a < (codec ? 0 : L::KATOMS); ++a)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(vst + L::LR_TILE + a * L::ATOM + tt * 128 + 16 * c) =
                    make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int c = 0; c < LSPAN / 16; ++c)
              *reinterpret_cast<uint4*>(vst + tt * LSPAN + 16 * c) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        tc::fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(PF + pb));
          if (!codec) mbar_arrive(bar(EMPTY + v));
        }
        prev_v = v;
        prev_vpar = (vi / NS) & 1;
        prev_tok = tok_ok;
        pending_v = codec;
      }
      if (pending_v) expand_v(prev_v, prev_vpar, prev_tok);

      // ---- this pipeline's split partial: m, l, O, O_lr of every row
      bool aborted = named_bar_or(bar_g, 128, failed);
      if (!aborted && i > 0) {
        const bool okp = wait_ab(bar(PR + pb), (i - 1) & 1, p.status, abort_flag);
        aborted = named_bar_or(bar_g, 128, !okp);
      }
      if (aborted) {
        if (tt == 0) *abort_flag = 1;
      } else {
        uint32_t o[kRows], ol[kRows];
        if (i > 0) {
          tc::fence_after();
          tc::ld_cols<kRows>(tl + ROT_COL + 16 * pb, o);
          tc::ld_cols<kRows>(tl + ROL_COL + 16 * pb, ol);
          tc::wait_ld();
        }
        float* rg = red + pb * 4 * kRows;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          float x = l_run[r];
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o2);
          if (lane == 0) rg[(warp & 3) * kRows + r] = x;
        }
        named_bar_sync(bar_g, 128);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          if (r < nrows) {
            const int64_t rec = rec_of(r, pb);
            float* po = p.part_o + rec * (D + R);
            if (tt < D) po[tt] = i > 0 ? __uint_as_float(o[r]) : 0.f;
            if (tt < R) po[D + tt] = (i > 0 && p.has_bv) ? __uint_as_float(ol[r]) : 0.f;
            if (tt == r) {
              p.part_ml[2 * rec] = m_run[r];
              p.part_ml[2 * rec + 1] = rg[r] + rg[kRows + r] + rg[2 * kRows + r] + rg[3 * kRows + r];
            }
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

// ---------------------------------------------------------------- combine
// Merges the splits of each (query, head) with log-sum-exp weights, applies
// the reordered V term O_lr B_V,a once, divides by l and stores bf16.
// One CTA per (query, head); thread t owns column t of the partial rows.
// The (m, l) pairs, column t of up to kCombineBatch splits and the B_V rows
// are requested together, so a merge of that many splits is one round trip.
struct CombineParams {
  const float* part_ml;
  const float* part_o;
  const int32_t* ctx_q_start;
  const int32_t* adapter_ids;
  const __nv_bfloat16* B_V;
  __nv_bfloat16* out;
  int32_t* status;
  int num_queries, num_ctx, Hq, Hkv, g, n_splits, n_adapters, has_bv;
  int covered_rows;  // rows per context the decode grid covers (n_chunks * rows per item)
  int codec;         // the base part was accumulated over rotated values: rotate the merged sum back
};

constexpr int kCombineBatch = 32;  // splits requested per round

template <int D, int R>
struct CombineShape {
  static constexpr int NCOL = D + R;
  static constexpr int NT = (NCOL + 31) / 32 * 32;  // threads: one per column
  static constexpr int NW = NT / 32;
};

template <int D, int R>
__global__ void __launch_bounds__(CombineShape<D, R>::NT) combine_kernel(const __grid_constant__ CombineParams p) {
  using C = CombineShape<D, R>;
  constexpr int NCOL = C::NCOL, NT = C::NT, NW = C::NW;
  __shared__ float w_s[256];  // the plan keeps n_splits <= 256
  __shared__ float red[NW];
  __shared__ float olr[R];
  __shared__ float orot[D];  // compressed pool: the merged base part before the rotation back
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int64_t pair = blockIdx.x;
  const int n = static_cast<int>(pair / p.Hq), m = static_cast<int>(pair % p.Hq);
  const int S = p.n_splits;
  // the context holding query n (ctx_q_start is non-decreasing): its row of
  // head m must lie inside the rows the decode grid covered, else no split
  // wrote a partial for it and the output is zero
  __shared__ int covered;
  if (tid == 0) {
    int lo = 0, hi = p.num_ctx;  // find the last c with ctx_q_start[c] <= n
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.ctx_q_start + mid) <= n) lo = mid;
      else hi = mid;
    }
    const int q0 = __ldg(p.ctx_q_start + lo), q1 = __ldg(p.ctx_q_start + lo + 1);
    const bool inside = q0 <= n && n < q1 && q0 >= 0 && q1 <= p.num_queries;
    covered = inside && (n - q0) * p.g + m % p.g < p.covered_rows;
    if (!covered) report(p.status, LRKV_ERR_INDEX);
  }
  __syncthreads();
  if (!covered) {
    if (tid < D) p.out[pair * D + tid] = __float2bfloat16_rn(0.f);
    return;
  }
  const int a = __ldg(p.adapter_ids + n);
  const bool bad = a < -1 || a >= p.n_adapters;
  const bool use_lr = p.has_bv && a >= 0 && !bad;
  if (bad && tid == 0 && m == 0) report(p.status, LRKV_ERR_INDEX);
  const float* ml = p.part_ml + pair * S * 2;
  const float* po = p.part_o + pair * S * NCOL + tid;
  // one round: (m, l) of split tid, column tid of the first splits, B_V rows
  float2 mlv = make_float2(-CUDART_INF_F, 0.f);
  if (tid < S) mlv = *reinterpret_cast<const float2*>(ml + 2 * tid);
  float pv[kCombineBatch];
#pragma unroll
  for (int s = 0; s < kCombineBatch; ++s) pv[s] = (tid < NCOL && s < S) ? po[static_cast<int64_t>(s) * NCOL] : 0.f;
  const __nv_bfloat16* bvp = p.B_V + (static_cast<int64_t>(use_lr ? a : 0) * R * p.Hkv + m / p.g) * D + tid;
  float bv[R];
#pragma unroll
  for (int k = 0; k < R; ++k) bv[k] = (use_lr && tid < D) ? __bfloat162float(bvp[static_cast<int64_t>(k) * p.Hkv * D]) : 0.f;
  // max over splits
  float M = mlv.x;
  for (int s = tid + NT; s < S; s += NT) M = fmaxf(M, ml[2 * s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) red[wid] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  // weights and the softmax denominator
  float Ls = 0.f;
  for (int s = tid; s < S; s += NT) {
    const float2 x = s == tid ? mlv : *reinterpret_cast<const float2*>(ml + 2 * s);
    const float w = (M == -CUDART_INF_F || x.x == -CUDART_INF_F) ? 0.f : exp2f(x.x - M);
    w_s[s] = w;
    Ls = fmaf(w, x.y, Ls);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
  if (lane == 0) red[wid] = Ls;
  __syncthreads();
  Ls = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) Ls += red[w];
  float v = 0.f;
  if (tid < NCOL) {
#pragma unroll
    for (int s = 0; s < kCombineBatch; ++s)
      if (s < S) v = fmaf(w_s[s], pv[s], v);
    // further splits: a batch of loads in flight, then its products
    for (int s0 = kCombineBatch; s0 < S; s0 += kCombineBatch) {
#pragma unroll
      for (int s = 0; s < kCombineBatch; ++s) pv[s] = s0 + s < S ? po[static_cast<int64_t>(s0 + s) * NCOL] : 0.f;
#pragma unroll
      for (int s = 0; s < kCombineBatch; ++s)
        if (s0 + s < S) v = fmaf(w_s[s0 + s], pv[s], v);
    }
    if (tid >= D) olr[tid - D] = use_lr ? v : 0.f;
    if (p.codec && tid < D) orot[tid] = v;
  }
  __syncthreads();
  if (p.codec && tid < D) {
    // O_base = (H / sqrt(d)) O_rot, H the Sylvester-Hadamard matrix: entry
    // (tid, i) is (-1)^popcount(tid & i)
    float acc = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; ++i) acc += (__popc(tid & i) & 1) ? -orot[i] : orot[i];
    v = acc * (1.0f / kSqrtD<D>);
  }
  if (tid < D) {
    if (use_lr) {
#pragma unroll
      for (int k = 0; k < R; ++k) v = fmaf(olr[k], bv[k], v);
    }
    const float inv = (Ls > 0.f && !bad) ? 1.f / Ls : 0.f;
    p.out[pair * D + tid] = __float2bfloat16_rn(v * inv);
  }
}

template <int D, int R>
lrkv_status run(const lrkv_config& cfg, const DecodeArgs& a, const DecodePlan& plan,
                void* workspace, cudaStream_t stream) {
  using L = DL<D, R>;
  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.ctx_q_start = a.ctx_q_start;
  p.adapter_ids = a.adapter_ids;
  p.block_tables = a.block_tables;
  p.ctx_lens = a.ctx_lens;
  p.B_K = static_cast<const __nv_bfloat16*>(a.B_K);
  p.B_V = static_cast<const __nv_bfloat16*>(a.B_V);
  const int64_t nrec = static_cast<int64_t>(a.num_queries) * cfg.n_q_heads * plan.n_splits * (plan.rebuild ? 2 : 1);
  p.part_ml = static_cast<float*>(workspace);
  p.part_o = p.part_ml + ((nrec * 2 + 63) / 64) * 64;
  p.status = a.status;
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks;
  p.max_ctx_len = a.max_ctx_len;
  p.n_adapters = a.n_adapters;
  p.num_queries = a.num_queries;
  p.Hq = cfg.n_q_heads;
  p.Hkv = cfg.n_kv_heads;
  p.g = plan.g;
  p.rpi = plan.rows_per_item;
  p.n_chunks = plan.n_chunks;
  p.n_splits = plan.n_splits;
  p.split_blocks = plan.split_blocks;
  p.has_bk = a.B_K != nullptr;
  p.has_bv = a.B_V != nullptr;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.lr_groups = cfg.lr_groups;
  p.test_stall = decode_test_stall();
  p.codec = cfg.kv_codec == LRKV_CODEC_POLYKV ? 1 : 0;
  p.cbase = static_cast<const uint8_t*>(a.base_pool);
  for (int k = 0; k < 8; ++k) p.vcent[k] = polykv_codec().centroid[k];
  rope_freqs(cfg, &p.freqs);

  CUtensorMap tb{}, tl, tk{};
  // a compressed base pool is read with plain bulk copies (no tensor map)
  if (!p.codec && !make_pool_maps(cfg, a.base_pool, nullptr, a.num_blocks, &tb, nullptr)) return LRKV_ERR_CUDA;
  if (!make_lr_map(cfg, a.lr_pool, a.num_blocks, L::RP, &tl)) return LRKV_ERR_CUDA;
  // G mode copies each item's B_K rows with a tensor map
  if (!plan.rebuild && p.has_bk && !make_bk_map(cfg, a.B_K, a.n_adapters, &tk)) return LRKV_ERR_CUDA;

  if (plan.n_items > 0) {
    auto kern = !plan.rebuild ? decode_kernel<D, R> : p.codec ? decode_rb_kernel<D, R, true> : decode_rb_kernel<D, R, false>;
    if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), plan.smem_bytes)) return LRKV_ERR_CUDA;
    kern<<<static_cast<unsigned>(plan.n_items), kThreads, plan.smem_bytes, stream>>>(p, tb, tl, tk);
    if (cudaGetLastError() != cudaSuccess) return LRKV_ERR_CUDA;
  }
  CombineParams c{};
  c.part_ml = p.part_ml;
  c.part_o = p.part_o;
  c.ctx_q_start = a.ctx_q_start;
  c.num_ctx = a.num_ctx;
  c.covered_rows = plan.n_chunks * plan.rows_per_item;
  c.adapter_ids = a.adapter_ids;
  c.B_V = static_cast<const __nv_bfloat16*>(a.B_V);
  c.out = static_cast<__nv_bfloat16*>(a.out);
  c.status = a.status;
  c.num_queries = a.num_queries;
  c.Hq = cfg.n_q_heads;
  c.Hkv = cfg.n_kv_heads;
  c.g = plan.g;
  c.n_splits = plan.n_splits * (plan.rebuild ? 2 : 1);  // rebuild mode: one partial per pipeline
  c.n_adapters = a.n_adapters;
  c.has_bv = a.B_V != nullptr;
  c.codec = p.codec;
  const int64_t pairs = static_cast<int64_t>(a.num_queries) * cfg.n_q_heads;
  if (pairs > 0) {
    // A plain stream-ordered launch: on this part, waiting resident on the
    // decode grid (programmatic dependent launch) released later than this.
    combine_kernel<D, R><<<static_cast<unsigned>(pairs), CombineShape<D, R>::NT, 0, stream>>>(c);
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
  // Rebuild mode (decode_rb_kernel) at rank 64, four rows per item: when every
  // item's rows belong to one query -- a multiple of 4 query heads per kv head,
  // or one query per context.
  P.rebuild = (R == 64 && (P.g % 4 == 0 || max_q_per_ctx == 1)) ? 1 : 0;
  // A compressed base pool is read by the rebuild-mode kernel only (it expands
  // the codes where it rebuilds K_a), at every rank; its items hold rows of one
  // query: up to 4 of them, a divisor of g unless each context has one query.
  int rb_rows = 4;
  if (cfg.kv_codec == LRKV_CODEC_POLYKV) {
    P.rebuild = 1;
    if (max_q_per_ctx > 1)
      while (P.g % rb_rows != 0) --rb_rows;
  }
  int rpi = 0, total = 0;
#define LRKV_L(d, r) \
  if (D == d && R == r) { rpi = DL<d, r>::RPI; total = DL<d, r>::total; }
  LRKV_L(128, 8) LRKV_L(128, 16) LRKV_L(128, 32) LRKV_L(128, 64)
  LRKV_L(64, 8) LRKV_L(64, 16) LRKV_L(64, 32) LRKV_L(64, 64)
#undef LRKV_L
  if (rpi == 0) return false;
  if (cfg.lr_groups > 1 && !P.rebuild) {
    // agent-specific A: an item's rows must belong to one query (one adapter,
    // one low-rank group): a query's heads of the kv head, or a part of them
    if (P.g <= rpi) rpi = P.g;
    else if (P.g % rpi != 0) return false;
  }
  if (P.rebuild) {
    rpi = rb_rows;
#define LRKV_RB(d, r) \
  if (D == d && R == r) total = rb::Layout<d, r>::total;
    LRKV_RB(128, 8) LRKV_RB(128, 16) LRKV_RB(128, 32) LRKV_RB(128, 64)
    LRKV_RB(64, 8) LRKV_RB(64, 16) LRKV_RB(64, 32) LRKV_RB(64, 64)
#undef LRKV_RB
  }
  P.rows_per_item = rpi;
  P.smem_bytes = std::max(total, kMinSmem);
  P.n_chunks = std::max(1, (max_q_per_ctx * P.g + rpi - 1) / rpi);
  const int nblk = std::max(1, (max_ctx_len + kBlock - 1) / kBlock);
  const int64_t pairs = static_cast<int64_t>(num_ctx) * P.n_chunks * cfg.n_kv_heads;
  // Splits: one CTA per item, one CTA per SM. Estimated time = waves x (blocks
  // per split + a per-item overhead of about 12 blocks' worth of streaming).
  constexpr double kItemOverheadBlocks = 12.0;
  int best_s = 1;
  double best = -1.0;
  // the combine kernel holds up to 256 split weights (rebuild mode: two partials per split)
  const int smax = std::min(nblk, P.rebuild ? 128 : 256);
  for (int s = 1; s <= smax; ++s) {
    const int sb = (nblk + s - 1) / s;
    if ((nblk + sb - 1) / sb != s) continue;
    const int64_t items = pairs * s;
    const int64_t waves = (items + sm_count - 1) / sm_count;
    const double cost = static_cast<double>(waves) * (sb + kItemOverheadBlocks);
    if (best < 0.0 || cost < best - 1e-9) {
      best = cost;
      best_s = s;
    }
  }
  P.split_blocks = (nblk + best_s - 1) / best_s;
  P.n_splits = (nblk + P.split_blocks - 1) / P.split_blocks;
  P.n_items = pairs * P.n_splits;
  if (P.n_items > INT32_MAX) return false;
  const int64_t nrec = static_cast<int64_t>(num_queries) * cfg.n_q_heads * P.n_splits * (P.rebuild ? 2 : 1);
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
