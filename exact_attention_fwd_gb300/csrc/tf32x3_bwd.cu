// tf32x3_bwd.cu — float32 attention backward on the tensor cores (3xTF32).
//
// Algorithm: "Flash Attention 2 — backward pass notes", section "The math (FA2
// backward with recompute)": with the saved L, P = exp(S - L) is recomputed;
// dP = dO V^T, dS = P (dP - D) with D = <dO, O>, dV = P^T dO,
// dK = scale dS^T Q, dQ = scale dS K; split as that page's option 3 ("Why the
// WGSL kernel isn't shipped this turn"): a kernel whose CTA owns 128 queries
// and writes dQ, and one whose CTA owns 128 keys and writes dK and dV, so
// every output row is written once (no atomics).  D comes from the float32 O
// (the pre-pass of bwd_dot.cu), so no correction is needed here.
//
// Every product is taken in 3xTF32 (tf32x3_common.cuh): hi*hi + hi*lo + lo*hi
// with tcgen05 kind::tf32 MMAs, fp32 accumulation in TMEM.  tf32 operands are
// K-major, so besides the hi / lo copies of Q, K, V, dO ([B, N, H, d]) the
// split pass writes transposed hi / lo copies of the tensors that are
// contracted over their rows: Q^T and dO^T (for dK and dV), K^T (for dQ), as
// [B, H, d, Np].
//
// One CTA per (b, h, 128-row tile), 8 warps:
//   warp 0 lane 0   TMA: the resident row tiles R1, R2 (hi, lo) once; per
//                   32-row streamed block, ring A (C1, C2 hi / lo: the
//                   operands of S and dP, freed when those MMAs complete) and
//                   ring B (the transposed operands of the accumulations,
//                   freed when they complete);
//   warps 1, 7      MMAs (lane 0): S = R1 C1^T (warp 1) and dP = R2 C2^T
//                   (warp 7), 24 MMAs each, M = 128, N = 32, fp32 in TMEM;
//   warp 6 lane 0   MMAs: the accumulations from the hi / lo element-wise
//                   results in TMEM (12 MMAs each, N = 64); three issuing
//                   threads, since one thread's issue rate bounds these
//                   N = 32 / 64 MMA streams;
//   warps 2-5       one thread per owned row (TMEM lane): P = 2^(S c - L2),
//                   dS = P (dP - D), masks, hi / lo split into TMEM; finally
//                   the accumulators, scaled, as float32 rows.
//   dQ kernel:    R1 = Q, R2 = dO, C1 = K, C2 = V, ring B = K^T;
//                 acc1 = dS K.
//   dK/dV kernel: R1 = K, R2 = V, C1 = Q, C2 = dO, ring B = Q^T, dO^T;
//                 acc1 = P^T dO (dV), acc2 = dS^T Q (dK).
// Shared memory: R1, R2 hi / lo 4 x 32 KB; ring A one slot of 32 KB (it is
// freed early, by the S / dP MMAs); ring B two slots (16 or 32 KB each).
// TMEM: S [0, 32), dP [32, 64), acc1 [64, 128), acc2 [128, 192), the first
// element-wise result hi / lo [192, 256), the second hi / lo [256, 320).
// Every wait is bounded (FA_ERR_TIMEOUT, abort flag, drain), as elsewhere.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <cmath>
#include <cstdint>

#include "fa_common.cuh"
#include "sm103_ptx.cuh"
#include "tf32x3_common.cuh"
#include "tmap.h"

namespace fa {
namespace {

constexpr int kRows = 128;               // rows owned by a CTA
constexpr int kBlk = 32;                 // rows of a streamed block
constexpr int kDP = 64;                  // padded head dim (d <= 64)
constexpr int kThreads = 256;
constexpr int kRChunk = kRows * 128;     // 32 fp32 columns of 128 rows (16 KB)
constexpr int kRTile = 2 * kRChunk;      // 128 x 64 fp32 (32 KB)
constexpr int kCChunk = kBlk * 128;      // 32 fp32 columns of 32 rows (4 KB)
constexpr int kCTile = 2 * kCChunk;      // 32 x 64 fp32 (8 KB)
constexpr int kTTile = kDP * 128;        // transposed: 64 rows (d) x 32 fp32 (8 KB)
constexpr int kASlot = 4 * kCTile;       // C1 hi, C1 lo, C2 hi, C2 lo
constexpr int kBSlots = 2;
constexpr int kBSlot = 4 * kTTile;       // up to two transposed pairs (hi, lo)
constexpr int kOffR = 0;                 // R1 hi, R1 lo, R2 hi, R2 lo
constexpr int kOffA = 4 * kRTile;
constexpr int kOffB = kOffA + kASlot;
constexpr int kOffBar = kOffB + kBSlots * kBSlot;
constexpr int kSmemBytes = kOffBar + 256 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per block");
constexpr int kTmemCols = 512;
constexpr uint32_t kColS = 0, kColdP = 32, kColAcc1 = 64, kColAcc2 = 128;
constexpr uint32_t kColXh = 192, kColXl = 224, kColYh = 256, kColYl = 288;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdTf32Bars {
  uint64_t r_full;
  uint64_t a_full, a_empty;
  uint64_t b_full[kBSlots], b_empty[kBSlots];
  uint64_t sp_full, sp_free, x_full, acc_done, acc_full, drain, probe;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void bt_abort(BwdTf32Bars* bars, int* status) {
  record_error(status, FA_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&bars->abort) = 1;
}

// A tile's streamed blocks: [first, first + count) in units of kBlk rows.
struct Span {
  int first, count;
};

// dQ kernel, query tile qt: the key blocks it reads (causal: up to the
// tile's last query).  dK/dV kernel, key tile kt: the query blocks that see
// one of its keys (causal: from the tile's first key on).
template <bool kDkDv, bool kCausal>
__device__ __forceinline__ Span span_of(int tile, int N) {
  const int nblk = (N + kBlk - 1) / kBlk;
  if constexpr (kDkDv) {
    const int first = kCausal ? (tile * kRows) / kBlk : 0;
    return Span{first, nblk - first};
  } else {
    const int last_row = min(N, (tile + 1) * kRows) - 1;
    return Span{0, kCausal ? min(nblk, last_row / kBlk + 1) : nblk};
  }
}

// 8 K-steps of 8 tf32 (32 bytes) over a 2-chunk K-major tile, or 4 over a
// 1-chunk tile: descriptor start-address offsets in 16-byte units.
__device__ __forceinline__ uint64_t ks(int kk, int chunk_bytes) { return kstep(kk, chunk_bytes); }

template <bool kDkDv, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tf32x3_kernel(const __grid_constant__ CUtensorMap tmR1h,
                      const __grid_constant__ CUtensorMap tmR1l,
                      const __grid_constant__ CUtensorMap tmR2h,
                      const __grid_constant__ CUtensorMap tmR2l,
                      const __grid_constant__ CUtensorMap tmC1h,
                      const __grid_constant__ CUtensorMap tmC1l,
                      const __grid_constant__ CUtensorMap tmC2h,
                      const __grid_constant__ CUtensorMap tmC2l,
                      const __grid_constant__ CUtensorMap tmT1h,
                      const __grid_constant__ CUtensorMap tmT1l,
                      const __grid_constant__ CUtensorMap tmT2h,
                      const __grid_constant__ CUtensorMap tmT2l, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  BwdTf32Bars* bars = reinterpret_cast<BwdTf32Bars*>(smem + kOffBar);
  const volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int N = p.N, H = p.H;
  const int nt = (N + kRows - 1) / kRows;
  const int tile = blockIdx.x % nt, bh = blockIdx.x / nt;
  const int b = bh / H, h = bh % H;
  const Span span = span_of<kDkDv, kCausal>(tile, N);
  const int nb = span.count;
  constexpr int kTPairs = kDkDv ? 2 : 1;   // transposed (hi, lo) pairs per ring-B slot

  if (threadIdx.x == 0) {
    mbar_init(&bars->r_full, 1);
    mbar_init(&bars->a_full, 1);
    mbar_init(&bars->a_empty, 2);   // S and dP issuers
    for (int s = 0; s < kBSlots; ++s) {
      mbar_init(&bars->b_full[s], 1);
      mbar_init(&bars->b_empty[s], 1);
    }
    mbar_init(&bars->sp_full, 2);   // S and dP issuers
    mbar_init(&bars->sp_free, kRows);
    mbar_init(&bars->x_full, kRows);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->drain, 3);   // one commit per MMA warp
    mbar_init(&bars->probe, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool run = true;
  if (p.probe_timeout) {
    // self-test of the bounded-wait path: nothing ever arrives on `probe`
    if (threadIdx.x == 0 && !mbar_wait(&bars->probe, 0, abort_flag, kProbeBudget))
      bt_abort(bars, p.status);
    __syncthreads();
    run = false;
  }
  uint8_t* sR = smem + kOffR;   // R1 hi, R1 lo, R2 hi, R2 lo
  uint8_t* sA = smem + kOffA;   // C1 hi, C1 lo, C2 hi, C2 lo
  auto bslot = [&](int s) { return smem + kOffB + s * kBSlot; };   // T1 hi, lo (, T2 hi, lo)

  if (run && warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      const CUtensorMap* rmaps[4] = {&tmR1h, &tmR1l, &tmR2h, &tmR2l};
      const CUtensorMap* cmaps[4] = {&tmC1h, &tmC1l, &tmC2h, &tmC2l};
      const CUtensorMap* tmaps[4] = {&tmT1h, &tmT1l, &tmT2h, &tmT2l};
      mbar_arrive_expect_tx(&bars->r_full, 4 * kRTile);
      for (int t = 0; t < 4; ++t)
        for (int ch = 0; ch < 2; ++ch)
          tma_load_4d(sR + t * kRTile + ch * kRChunk, rmaps[t], &bars->r_full, ch * 32, h,
                      tile * kRows, b);
      bool ok = true;
      int i = 0;
      for (; i < nb; ++i) {
        const int blk = span.first + i;
        // ring A (one slot): the S / dP operands of block i
        if (i > 0 && !mbar_wait(&bars->a_empty, (i - 1) & 1, abort_flag, kWaitBudget)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars->a_full, kASlot);
        for (int t = 0; t < 4; ++t)
          for (int ch = 0; ch < 2; ++ch)
            tma_load_4d(sA + t * kCTile + ch * kCChunk, cmaps[t], &bars->a_full, ch * 32, h,
                        blk * kBlk, b);
        // ring B (two slots): the transposed operands of block i's accumulations
        const int s = i % kBSlots;
        if (i >= kBSlots &&
            !mbar_wait(&bars->b_empty[s], (i / kBSlots - 1) & 1, abort_flag, kWaitBudget)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars->b_full[s], kTPairs * 2 * kTTile);
        for (int t = 0; t < 2 * kTPairs; ++t)
          tma_load_4d(bslot(s) + t * kTTile, tmaps[t], &bars->b_full[s], blk * kBlk, 0, h, b);
      }
      if (!ok) bt_abort(bars, p.status);
      // every issued copy has landed before the CTA may exit
      mbar_wait(&bars->r_full, 0, nullptr, kDrainBudget);
      if (i > 0) mbar_wait(&bars->a_full, (i - 1) & 1, nullptr, kDrainBudget);
      for (int x = (i > kBSlots ? i - kBSlots : 0); x < i; ++x)
        mbar_wait(&bars->b_full[x % kBSlots], (x / kBSlots) & 1, nullptr, kDrainBudget);
    }
    __syncwarp();
  }
  else if (run && (warp == 1 || warp == 6 || warp == 7)) {
    // ====== MMA issuers (whole warp waits, lane 0 issues): warp 1 S, warp 7 dP, warp 6 the accumulations ======
    const bool leader = lane == 0;
    constexpr uint32_t kIdescSP = idesc_tf32(kRows, kBlk);   // S, dP: N = 32 streamed rows
    constexpr uint32_t kIdescAcc = idesc_tf32(kRows, kDP);   // accumulations: N = 64 columns
    const uint64_t dR1h = sdesc_sw128(smem_u32(sR), 16, 1024);
    const uint64_t dR1l = sdesc_sw128(smem_u32(sR + kRTile), 16, 1024);
    const uint64_t dR2h = sdesc_sw128(smem_u32(sR + 2 * kRTile), 16, 1024);
    const uint64_t dR2l = sdesc_sw128(smem_u32(sR + 3 * kRTile), 16, 1024);
    const uint64_t dC1h = sdesc_sw128(smem_u32(sA), 16, 1024);
    const uint64_t dC1l = sdesc_sw128(smem_u32(sA + kCTile), 16, 1024);
    const uint64_t dC2h = sdesc_sw128(smem_u32(sA + 2 * kCTile), 16, 1024);
    const uint64_t dC2l = sdesc_sw128(smem_u32(sA + 3 * kCTile), 16, 1024);
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->r_full, 0, abort_flag, kWaitBudget));
    // S = R1 C1^T and dP = R2 C2^T of block i (3xTF32 each, K = the head dim:
    // columns >= d are zero-filled, so 8 K-steps are exact for every d <= 64)
    auto issue_sp = [&](int i) -> bool {
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&bars->a_full, i & 1, abort_flag, kWaitBudget) &&
                          (i == 0 ||
                           mbar_wait(&bars->sp_free, (i - 1) & 1, abort_flag, kWaitBudget))))
        return false;
      tc_fence_after();
      if (leader && warp == 1) {
#pragma unroll
        for (int kk = 0; kk < kDP / 8; ++kk)
          mma_ss_tf32(tmem + kColS, dR1h + ks(kk, kRChunk), dC1h + ks(kk, kCChunk), kIdescSP,
                      kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kDP / 8; ++kk)
          mma_ss_tf32(tmem + kColS, dR1h + ks(kk, kRChunk), dC1l + ks(kk, kCChunk), kIdescSP, 1u);
#pragma unroll
        for (int kk = 0; kk < kDP / 8; ++kk)
          mma_ss_tf32(tmem + kColS, dR1l + ks(kk, kRChunk), dC1h + ks(kk, kCChunk), kIdescSP, 1u);
      }
      if (leader && warp == 7) {
#pragma unroll
        for (int kk = 0; kk < kDP / 8; ++kk)
          mma_ss_tf32(tmem + kColdP, dR2h + ks(kk, kRChunk), dC2h + ks(kk, kCChunk), kIdescSP,
                      kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kDP / 8; ++kk)
          mma_ss_tf32(tmem + kColdP, dR2h + ks(kk, kRChunk), dC2l + ks(kk, kCChunk), kIdescSP, 1u);
#pragma unroll
        for (int kk = 0; kk < kDP / 8; ++kk)
          mma_ss_tf32(tmem + kColdP, dR2l + ks(kk, kRChunk), dC2h + ks(kk, kCChunk), kIdescSP, 1u);
      }
      if (leader) {
        mma_commit(&bars->sp_full);
        mma_commit(&bars->a_empty);
      }
      __syncwarp();
      return true;
    };
    // acc += X T (hi*hi + hi*lo + lo*hi), X the element-wise result at
    // columns xh / xl of TMEM, T a transposed (d x 32) pair in shared memory
    auto acc3 = [&](uint32_t acc, uint32_t xh, uint32_t xl, uint64_t th, uint64_t tl,
                    bool first) {
#pragma unroll
      for (int kk = 0; kk < kBlk / 8; ++kk)
        mma_ts_tf32(tmem + acc, tmem + xh + kk * 8, th + ks(kk, kTTile), kIdescAcc,
                    (!first || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < kBlk / 8; ++kk)
        mma_ts_tf32(tmem + acc, tmem + xh + kk * 8, tl + ks(kk, kTTile), kIdescAcc, 1u);
#pragma unroll
      for (int kk = 0; kk < kBlk / 8; ++kk)
        mma_ts_tf32(tmem + acc, tmem + xl + kk * 8, th + ks(kk, kTTile), kIdescAcc, 1u);
    };
    auto issue_acc = [&](int i) -> bool {
      const int s = i % kBSlots;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&bars->x_full, i & 1, abort_flag, kWaitBudget) &&
                          mbar_wait(&bars->b_full[s], (i / kBSlots) & 1, abort_flag,
                                    kWaitBudget)))
        return false;
      tc_fence_after();
      if (leader) {
        uint8_t* bs = bslot(s);
        const uint64_t dT1h = sdesc_sw128(smem_u32(bs), 16, 1024);
        const uint64_t dT1l = sdesc_sw128(smem_u32(bs + kTTile), 16, 1024);
        if constexpr (kDkDv) {
          const uint64_t dT2h = sdesc_sw128(smem_u32(bs + 2 * kTTile), 16, 1024);
          const uint64_t dT2l = sdesc_sw128(smem_u32(bs + 3 * kTTile), 16, 1024);
          acc3(kColAcc1, kColXh, kColXl, dT2h, dT2l, i == 0);   // dV += P^T dO
          acc3(kColAcc2, kColYh, kColYl, dT1h, dT1l, i == 0);   // dK += dS^T Q
        } else {
          acc3(kColAcc1, kColXh, kColXl, dT1h, dT1l, i == 0);   // dQ += dS K
        }
        mma_commit(&bars->acc_done);
        mma_commit(&bars->b_empty[s]);
        if (i == nb - 1) mma_commit(&bars->acc_full);
      }
      __syncwarp();
      return true;
    };
    if (warp != 6) {
      for (int i = 0; i < nb && ok; ++i)
        if (!issue_sp(i)) ok = false;
    } else {
      for (int i = 0; i < nb && ok; ++i)
        if (!issue_acc(i)) ok = false;
    }
    if (!ok && leader) bt_abort(bars, p.status);
    // no MMA may be in flight when TMEM is released
    mma_commit_w(&bars->drain, leader ? 1u : 0u);
    mbar_wait(&bars->drain, 0, nullptr, kDrainBudget);
    __syncwarp();
  }
  else if (run && warp >= 2 && warp <= 5) {
    // ============ element-wise warps 2-5: one thread per owned row ============
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
    const int grow = tile * kRows + row;   // owned query (dQ) or key (dK/dV)
    const size_t hb = static_cast<size_t>(bh) * N;
    const float c = p.scale_log2;
    // dQ kernel: the owned query's L (base 2) and D; a padded or fully
    // masked query (L = -inf) gets 2^-inf = 0 everywhere
    float l2_row = INFINITY, d_row = 0.0f;
    if (!kDkDv && grow < N) {
      const float L = p.lse[hb + grow];
      if (L != -INFINITY) {
        l2_row = L * kLog2e;
        d_row = p.D[hb + grow];
      }
    }
    bool ok = true;
    for (int i = 0; i < nb; ++i) {
      const int col0 = (span.first + i) * kBlk;   // first streamed row: key (dQ) / query (dK/dV)
      // dK/dV: the block's per-query L (base 2) and D (the same for every row)
      float l2c[kBlk], dc[kBlk];
      if constexpr (kDkDv) {
#pragma unroll
        for (int j = 0; j < kBlk; ++j) {
          const int q = col0 + j;
          float L = -INFINITY, dd = 0.0f;
          if (q < N) {
            L = p.lse[hb + q];
            dd = p.D[hb + q];
          }
          l2c[j] = (L == -INFINITY) ? INFINITY : L * kLog2e;
          dc[j] = (L == -INFINITY) ? 0.0f : dd;
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->sp_full, i & 1, abort_flag, kWaitBudget))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[kBlk], dr[kBlk];
      tmem_ld32(tmem + lb + kColS, sr);
      tmem_ld32(tmem + lb + kColdP, dr);
      tmem_ld_wait(sr);
      tmem_ld_wait(dr);
      tc_fence_before();
      mbar_arrive(&bars->sp_free);   // S and dP may take the next block's scores
      uint32_t xh[kBlk], xl[kBlk], yh[kBlk], yl[kBlk];
      // masked pairs: P = 0 (dQ: key beyond N or after the query; dK/dV:
      // query before the key; queries beyond N carry L2 = +inf), as one keep
      // bit per column of the block
      uint32_t keep;
      if constexpr (kDkDv) {
        const int sh = kCausal ? grow - col0 : 0;   // keep columns sh ..
        keep = sh <= 0 ? 0xffffffffu : (sh >= 32 ? 0u : (0xffffffffu << sh));
      } else {
        const int lim = (kCausal ? min(grow, N - 1) : N - 1) - col0;   // keep columns .. lim
        keep = lim >= 31 ? 0xffffffffu : (lim < 0 ? 0u : (0xffffffffu >> (31 - lim)));
      }
#pragma unroll
      for (int j = 0; j < kBlk; ++j) {
        const bool masked = ((keep >> j) & 1u) == 0u;
        const float l2 = kDkDv ? l2c[j] : l2_row;
        const float dd = kDkDv ? dc[j] : d_row;
        const float pv = masked ? 0.0f : fast_exp2(__uint_as_float(sr[j]) * c - l2);
        const float ds = pv * (__uint_as_float(dr[j]) - dd);
        const float x = kDkDv ? pv : ds;   // the operand of acc1
        const float xhi = tf32_rn(x);
        xh[j] = __float_as_uint(xhi);
        xl[j] = __float_as_uint(tf32_rn(x - xhi));
        if constexpr (kDkDv) {
          const float dhi = tf32_rn(ds);
          yh[j] = __float_as_uint(dhi);
          yl[j] = __float_as_uint(tf32_rn(ds - dhi));
        }
      }
      // the previous block's accumulations have read the element-wise columns
      if (i > 0 &&
          !__all_sync(0xffffffffu, mbar_wait(&bars->acc_done, (i - 1) & 1, abort_flag,
                                             kWaitBudget))) {
        ok = false;
        break;
      }
      tc_fence_after();
      __syncwarp();   // tcgen05.st is warp-collective
      tmem_st32(tmem + lb + kColXh, xh);
      tmem_st32(tmem + lb + kColXl, xl);
      if constexpr (kDkDv) {
        tmem_st32(tmem + lb + kColYh, yh);
        tmem_st32(tmem + lb + kColYl, yl);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->x_full);
    }
    if (ok && nb > 0 &&
        !__all_sync(0xffffffffu, mbar_wait(&bars->acc_full, 0, abort_flag, kWaitBudget)))
      ok = false;
    if (ok) {
      // ---- epilogue: the accumulators, scaled, as float32 rows ----
      tc_fence_after();
      const bool store = grow < N;
      const size_t roff = ((static_cast<size_t>(b) * N + (store ? grow : 0)) * H + h) *
                          static_cast<size_t>(p.d);
      auto store_acc = [&](uint32_t acc, float mul, float* out) {
#pragma unroll
        for (int cc = 0; cc < kDP / 32; ++cc) {
          uint32_t a[32];
          __syncwarp();   // tcgen05.ld is warp-collective
          tmem_ld32(tmem + lb + acc + cc * 32, a);
          tmem_ld_wait(a);
          if (store) {
#pragma unroll
            for (int qv = 0; qv < 8; ++qv) {
              const int col = cc * 32 + qv * 4;
              if (col < p.d)
                *reinterpret_cast<float4*>(out + roff + col) =
                    make_float4(__uint_as_float(a[qv * 4 + 0]) * mul,
                                __uint_as_float(a[qv * 4 + 1]) * mul,
                                __uint_as_float(a[qv * 4 + 2]) * mul,
                                __uint_as_float(a[qv * 4 + 3]) * mul);
            }
          }
        }
      };
      if constexpr (kDkDv) {
        store_acc(kColAcc1, 1.0f, static_cast<float*>(p.dv));
        store_acc(kColAcc2, p.scale, static_cast<float*>(p.dk));
      } else {
        store_acc(kColAcc1, p.scale, static_cast<float*>(p.dq));
      }
    } else {
      bt_abort(bars, p.status);
    }
    tc_fence_before();
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

namespace {

int round4_b(int n) { return (n + 3) & ~3; }
size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

// Workspace: D [B, H, N]; the hi / lo copies of Q, K, V, dO ([B, N, H, d]);
// the transposed hi / lo copies of Q, K, dO ([B, H, d, Np]); every part
// rounded up to 256 bytes.
size_t tf32x3_bwd_workspace_bytes(int B, int H, int N, int d) {
  const size_t db = round256(static_cast<size_t>(B) * H * N * 4);
  const size_t a = round256(static_cast<size_t>(B) * N * H * d * 4);
  const size_t t = round256(static_cast<size_t>(B) * H * d * round4_b(N) * 4);
  return db + 8 * a + 6 * t;
}

cudaError_t launch_bwd_tf32x3(const BwdParams& p_in, void* workspace, cudaStream_t st,
                              bool causal) {
  const int B = p_in.B, H = p_in.H, N = p_in.N, d = p_in.d, Np = round4_b(N);
  if (d > kDP || d % 8 != 0) return cudaErrorNotSupported;
  const size_t db = round256(static_cast<size_t>(B) * H * N * 4);
  const size_t a = round256(static_cast<size_t>(B) * N * H * d * 4);
  const size_t t = round256(static_cast<size_t>(B) * H * d * Np * 4);
  char* w = static_cast<char*>(workspace);
  BwdParams p = p_in;
  p.D = reinterpret_cast<float*>(w);
  float* split[8];   // Qh Ql Kh Kl Vh Vl dOh dOl
  for (int i = 0; i < 8; ++i) split[i] = reinterpret_cast<float*>(w + db + i * a);
  float* tsplit[6];  // QTh QTl KTh KTl dOTh dOTl
  for (int i = 0; i < 6; ++i) tsplit[i] = reinterpret_cast<float*>(w + db + 8 * a + i * t);

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return cudaErrorInvalidDevice;
  // split passes: B N H d is a multiple of 4 (d is a multiple of 8) and the
  // inputs are 16-byte aligned
  const size_t n4 = static_cast<size_t>(B) * N * H * d / 4;
  const size_t want = (n4 + 255) / 256, cap = static_cast<size_t>(sms) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  split_qk_kernel<<<grid, 256, 0, st>>>(
      static_cast<const float4*>(p.q), static_cast<const float4*>(p.k),
      reinterpret_cast<float4*>(split[0]), reinterpret_cast<float4*>(split[1]),
      reinterpret_cast<float4*>(split[2]), reinterpret_cast<float4*>(split[3]), n4);
  split_qk_kernel<<<grid, 256, 0, st>>>(
      static_cast<const float4*>(p.v), static_cast<const float4*>(p.dO),
      reinterpret_cast<float4*>(split[4]), reinterpret_cast<float4*>(split[5]),
      reinterpret_cast<float4*>(split[6]), reinterpret_cast<float4*>(split[7]), n4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (static_cast<long long>(B) * H > 65535) return cudaErrorInvalidConfiguration;
  const dim3 tgrid((Np + 31) / 32, (d + 63) / 64, B * H);
  const float* tsrc[3] = {static_cast<const float*>(p.q), static_cast<const float*>(p.k),
                          static_cast<const float*>(p.dO)};
  for (int i = 0; i < 3; ++i)
    split_vt_kernel<<<tgrid, 256, 0, st>>>(tsrc[i], tsplit[2 * i], tsplit[2 * i + 1], N, H, d, Np);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // D = rowsum(dO * O) from the float32 O
  e = launch_bwd_dot(p, 0, st);
  if (e != cudaSuccess) return e;

  // tensor maps: [B, N, H, d] as (d, H, N, B); transposed [B, H, d, Np] as (Np, d, H, B)
  const cuuint64_t dn[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                            static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
  const cuuint64_t sn[3] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(H) * d * 4,
                            static_cast<cuuint64_t>(N) * H * d * 4};
  const cuuint64_t dt[4] = {static_cast<cuuint64_t>(Np), static_cast<cuuint64_t>(d),
                            static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t stt[3] = {static_cast<cuuint64_t>(Np) * 4, static_cast<cuuint64_t>(d) * Np * 4,
                             static_cast<cuuint64_t>(H) * d * Np * 4};
  const cuuint32_t box_r[4] = {32u, 1u, static_cast<cuuint32_t>(kRows), 1u};
  const cuuint32_t box_c[4] = {32u, 1u, static_cast<cuuint32_t>(kBlk), 1u};
  const cuuint32_t box_t[4] = {32u, static_cast<cuuint32_t>(kDP), 1u, 1u};
  // R and C maps of the four split tensors, T maps of the three transposed ones
  CUtensorMap rm[8], cm[8], tm[6];
  for (int i = 0; i < 8 && e == cudaSuccess; ++i) {
    e = make_f32_tmap(&rm[i], split[i], dn, sn, box_r);
    if (e == cudaSuccess) e = make_f32_tmap(&cm[i], split[i], dn, sn, box_c);
  }
  for (int i = 0; i < 6 && e == cudaSuccess; ++i) e = make_f32_tmap(&tm[i], tsplit[i], dt, stt, box_t);
  if (e != cudaSuccess) return e;
  const long long ctas = static_cast<long long>(B) * H * ((N + kRows - 1) / kRows);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // index of each tensor in split[]: Q 0, K 2, V 4, dO 6; in tsplit[]: Q^T 0, K^T 2, dO^T 4
  auto launch = [&](auto kern, int r1, int r2, int c1, int c2, int t1, int t2) -> cudaError_t {
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    BwdParams pc = p;
    void* args[] = {&rm[r1], &rm[r1 + 1], &rm[r2], &rm[r2 + 1], &cm[c1], &cm[c1 + 1],
                    &cm[c2], &cm[c2 + 1], &tm[t1], &tm[t1 + 1], &tm[t2], &tm[t2 + 1], &pc};
    return cudaLaunchKernel(reinterpret_cast<const void*>(kern),
                            dim3(static_cast<unsigned>(ctas)), dim3(kThreads), args, kSmemBytes,
                            st);
  };
  // dQ: R1 = Q, R2 = dO, C1 = K, C2 = V, T1 = K^T
  e = causal ? launch(bwd_tf32x3_kernel<false, true>, 0, 6, 2, 4, 2, 2)
             : launch(bwd_tf32x3_kernel<false, false>, 0, 6, 2, 4, 2, 2);
  if (e != cudaSuccess) return e;
  // dK/dV: R1 = K, R2 = V, C1 = Q, C2 = dO, T1 = Q^T, T2 = dO^T
  return causal ? launch(bwd_tf32x3_kernel<true, true>, 2, 4, 0, 6, 0, 4)
                : launch(bwd_tf32x3_kernel<true, false>, 2, 4, 0, 6, 0, 4);
}

}  // namespace fa
