// tf32x3_fwd.cu — float32 attention forward on the tensor cores (3xTF32).
//
// Algorithm: "Flash Attention 2 — forward pass notes", sections "Loop (per
// (b, h, Q-tile))" and "What's still needed for full FA2" item 1, as in the
// 16-bit kernel; here every input and output is float32.
//
// tcgen05 kind::tf32 multiplies 32-bit operands with 10 explicit mantissa
// bits.  Each float32 x is split into hi = x rounded to the nearest tf32
// value and lo = (x - hi) rounded to the nearest tf32 value (x - hi is exact
// in float32 and |x - hi| <= 2^-11 |x|), and a product is taken as
// hi*hi + hi*lo + lo*hi.  The dropped lo*lo term and the two roundings of lo
// leave at most about 3 * 2^-22 relative error per product, and the operands
// are already tf32 values, so how the tensor cores reduce 32-bit operands to
// tf32 does not matter.
//
//   1. split pass (HBM-bound): Qh, Ql, Kh, Kl as [B, N, H, d] (16-byte
//      accesses) and V^T split as [B, H, d, Np] (Np = N rounded up to 4, zeros
//      beyond N; transposed through shared-memory tiles), so that every MMA
//      operand is K-major;
//   2. fused pass, one CTA per (b, h, 128-row Q tile), 8 warps:
//        warp 0 lane 0   TMA: Qh, Ql once; Kh, Kl of each key block into a
//                        ring that S frees;
//        warp 6 lane 0   TMA: V^Th, V^Tl of each block into a ring that P V
//                        frees (the K loads run ahead of the V releases);
//        warp 1 lane 0   MMAs: S = Qh Kh^T + Qh Kl^T + Ql Kh^T (fp32 in TMEM);
//        warp 7 lane 0   MMAs: O += Ph Vh + Ph Vl + Pl Vh (P read from TMEM);
//        warps 2-5       one thread per query row (TMEM lane): masked row max,
//                        lazy rescale, P = 2^(s c - m) in float32 split into
//                        Ph, Pl in TMEM; finally O / l and L.
// Head dims up to 64 use 64-key blocks, a 3-slot K ring and a 2-slot V ring;
// head dims up to 128 (the hi / lo Q tile then takes 128 KB) use 32-key
// blocks, 2 K slots and 1 V slot (T3Cfg).  TMEM: S, Ph, Pl (one block's
// keys each), then O (the padded head dim).  S(j+1) is computed while the
// softmax works on block j; PV(j) runs once P(j) is in TMEM.  Every wait is
// bounded (FA_ERR_TIMEOUT, abort flag, drain).
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

constexpr int kBM = 128;                  // query rows per CTA
constexpr int kThreads = 256;
constexpr int kQChunk = kBM * 128;        // 32 fp32 columns of 128 rows
constexpr int kTmemCols = 256;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kKStagesMax = 3, kVStagesMax = 2;

// Padded head dim DP = 64: 64-key blocks, K ring 3 slots, V ring 2.
// DP = 128: the hi / lo Q tile is 128 KB, so 32-key blocks, K ring 2 slots,
// V ring 1 (every slot holds 16 KB hi + 16 KB lo either way).
template <int DP>
struct T3Cfg {
  static constexpr int kDP = DP;
  static constexpr int kBN = DP == 64 ? 64 : 32;          // keys per block
  static constexpr int kKStages = DP == 64 ? 3 : 2;       // (Kh, Kl) ring, freed when S has read it
  static constexpr int kVStages = DP == 64 ? 2 : 1;       // (V^Th, V^Tl) ring, freed by P V
  static constexpr int kKChunk = kBN * 128;               // 32 fp32 columns of kBN rows
  static constexpr int kVChunk = DP * 128;                // 32 keys of V^T (DP rows)
  static constexpr int kQTile = (DP / 32) * kQChunk;      // 128 x DP fp32
  static constexpr int kKTile = kBN * DP * 4;             // kBN x DP (= V^T's DP x kBN)
  static constexpr int kOffQh = 0, kOffQl = kQTile;
  static constexpr int kPairBytes = 2 * kKTile;           // one ring slot: hi tile, then lo tile
  static constexpr int kOffK = 2 * kQTile;
  static constexpr int kOffV = kOffK + kKStages * kPairBytes;
  static constexpr int kOffBar = kOffV + kVStages * kPairBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per block");
  // TMEM: S [0, kBN), Ph [kBN, 2 kBN), Pl [2 kBN, 3 kBN), O [3 kBN, 3 kBN + DP)
  static constexpr uint32_t kColS = 0, kColPh = kBN, kColPl = 2 * kBN, kColO = 3 * kBN;
  static_assert(3 * kBN + DP <= kTmemCols, "TMEM columns");
};

struct Tf32Bars {
  uint64_t q_full;
  uint64_t k_full[kKStagesMax];
  uint64_t k_empty[kKStagesMax];
  uint64_t v_full[kVStagesMax];
  uint64_t v_empty[kVStagesMax];
  uint64_t s_full, s_free, p_full, pv_done, drain, probe;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void tf32_abort(Tf32Bars* bars, int* status) {
  record_error(status, FA_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&bars->abort) = 1;
}

template <int DP, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tf32x3_kernel(const __grid_constant__ CUtensorMap tmQh,
                      const __grid_constant__ CUtensorMap tmQl,
                      const __grid_constant__ CUtensorMap tmKh,
                      const __grid_constant__ CUtensorMap tmKl,
                      const __grid_constant__ CUtensorMap tmVh,
                      const __grid_constant__ CUtensorMap tmVl, const FwdParams p) {
  using Cfg = T3Cfg<DP>;
  constexpr int kBN = Cfg::kBN, kDP = Cfg::kDP, kKStages = Cfg::kKStages,
                kVStages = Cfg::kVStages, kKChunk = Cfg::kKChunk, kVChunk = Cfg::kVChunk,
                kQTile = Cfg::kQTile, kKTile = Cfg::kKTile, kPairBytes = Cfg::kPairBytes;
  constexpr int kOffQh = Cfg::kOffQh, kOffQl = Cfg::kOffQl, kOffK = Cfg::kOffK,
                kOffV = Cfg::kOffV, kOffBar = Cfg::kOffBar;
  constexpr uint32_t kColS = Cfg::kColS, kColPh = Cfg::kColPh, kColPl = Cfg::kColPl,
                     kColO = Cfg::kColO;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Tf32Bars* bars = reinterpret_cast<Tf32Bars*>(smem + kOffBar);
  const volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int N = p.N, H = p.H;
  const int nq = (N + kBM - 1) / kBM, nk = (N + kBN - 1) / kBN;
  const int qt = blockIdx.x % nq, bh = blockIdx.x / nq;
  const int b = bh / H, h = bh % H;
  // key blocks this tile visits (causal: up to its last row's diagonal)
  const int nb = kCausal ? min(nk, (min(N, (qt + 1) * kBM) - 1) / kBN + 1) : nk;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, kBM);
    mbar_init(&bars->p_full, kBM);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->drain, 2);   // one commit per MMA warp
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
      tf32_abort(bars, p.status);
    __syncthreads();
    run = false;
  }
  uint8_t* sQh = smem + kOffQh;
  uint8_t* sQl = smem + kOffQl;
  auto kslot = [&](int s) { return smem + kOffK + s * kPairBytes; };
  auto vslot = [&](int s) { return smem + kOffV + s * kPairBytes; };

  if (run && (warp == 0 || warp == 6)) {
    // ============ TMA producers: warp 0 loads Q and K, warp 6 loads V ============
    // (separate rings, so a K load never waits behind the release of a V slot)
    if (lane == 0) {
      const bool is_k = warp == 0;
      const int depth = is_k ? kKStages : kVStages;
      uint64_t* full = is_k ? bars->k_full : bars->v_full;
      uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
      bool ok = true;
      if (is_k) {
        mbar_arrive_expect_tx(&bars->q_full, 2 * kQTile);
        for (int ch = 0; ch < kDP / 32; ++ch) {
          tma_load_4d(sQh + ch * kQChunk, &tmQh, &bars->q_full, ch * 32, h, qt * kBM, b);
          tma_load_4d(sQl + ch * kQChunk, &tmQl, &bars->q_full, ch * 32, h, qt * kBM, b);
        }
      }
      int j = 0;
      for (; j < nb; ++j) {
        const int s = j % depth, round = j / depth;
        if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1, abort_flag, kWaitBudget)) {
          ok = false;
          break;
        }
        uint8_t* slot = is_k ? kslot(s) : vslot(s);
        mbar_arrive_expect_tx(&full[s], kPairBytes);
        if (is_k) {
          for (int ch = 0; ch < kDP / 32; ++ch) {
            tma_load_4d(slot + ch * kKChunk, &tmKh, &full[s], ch * 32, h, j * kBN, b);
            tma_load_4d(slot + kKTile + ch * kKChunk, &tmKl, &full[s], ch * 32, h, j * kBN, b);
          }
        } else {
          for (int ch = 0; ch < kBN / 32; ++ch) {
            tma_load_4d(slot + ch * kVChunk, &tmVh, &full[s], j * kBN + ch * 32, 0, h, b);
            tma_load_4d(slot + kKTile + ch * kVChunk, &tmVl, &full[s], j * kBN + ch * 32, 0, h, b);
          }
        }
      }
      if (!ok) tf32_abort(bars, p.status);
      // every issued copy has landed before the CTA may exit
      if (is_k) mbar_wait(&bars->q_full, 0, nullptr, kDrainBudget);
      for (int x = max(0, j - depth); x < j; ++x)
        mbar_wait(&full[x % depth], (x / depth) & 1, nullptr, kDrainBudget);
    }
    __syncwarp();
  }
  else if (run && (warp == 1 || warp == 7)) {
    // ===== MMA issuers (whole warp waits, lane 0 issues): warp 1 S, warp 7 P V =====
    // (one thread's issue rate bounds these N = 64 tf32 MMA streams, so the
    // two chains come from separate threads)
    const bool leader = lane == 0;
    constexpr uint32_t kIdescS = idesc_tf32(kBM, kBN);   // S: N = kBN keys
    constexpr uint32_t kIdescPV = idesc_tf32(kBM, kDP);  // PV: N = DP columns
    // K-steps over the padded head dim: columns >= d of Q and K are zero-filled
    // by the tensor maps, so a compile-time count (fully unrolled, constant
    // descriptor offsets) is exact for every d <= 64 and keeps the issuing
    // thread's instruction stream short.
    constexpr int nks = kDP / 8;
    const uint64_t dQh = sdesc_sw128(smem_u32(sQh), 16, 1024);
    const uint64_t dQl = sdesc_sw128(smem_u32(sQl), 16, 1024);
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full, 0, abort_flag, kWaitBudget));
    auto pv_step = [&](int jj) -> bool {   // O += Ph Vh + Ph Vl + Pl Vh of block jj
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&bars->p_full, jj & 1, abort_flag, kWaitBudget) &&
                          mbar_wait(&bars->v_full[jj % kVStages], (jj / kVStages) & 1, abort_flag,
                                    kWaitBudget)))
        return false;
      tc_fence_after();
      if (leader) {
        uint8_t* vs = vslot(jj % kVStages);
        const uint64_t dVh = sdesc_sw128(smem_u32(vs), 16, 1024);
        const uint64_t dVl = sdesc_sw128(smem_u32(vs + kKTile), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 8; ++kk)
          mma_ts_tf32(tmem + kColO, tmem + kColPh + kk * 8, dVh + kstep(kk, kVChunk), kIdescPV,
                      (jj > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kBN / 8; ++kk)
          mma_ts_tf32(tmem + kColO, tmem + kColPh + kk * 8, dVl + kstep(kk, kVChunk), kIdescPV, 1u);
#pragma unroll
        for (int kk = 0; kk < kBN / 8; ++kk)
          mma_ts_tf32(tmem + kColO, tmem + kColPl + kk * 8, dVh + kstep(kk, kVChunk), kIdescPV, 1u);
        mma_commit(&bars->pv_done);
        mma_commit(&bars->v_empty[jj % kVStages]);
      }
      __syncwarp();
      return true;
    };
    if (warp == 7) {
      for (int jj = 0; jj < nb && ok; ++jj)
        if (!pv_step(jj)) ok = false;
    }
    for (int j = 0; j < nb && ok && warp == 1; ++j) {
      const int s = j % kKStages;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&bars->k_full[s], (j / kKStages) & 1, abort_flag, kWaitBudget) &&
                          (j == 0 ||
                           mbar_wait(&bars->s_free, (j - 1) & 1, abort_flag, kWaitBudget)))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (leader) {
        uint8_t* ks = kslot(s);
        const uint64_t dKh = sdesc_sw128(smem_u32(ks), 16, 1024);
        const uint64_t dKl = sdesc_sw128(smem_u32(ks + kKTile), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < nks; ++kk)
          mma_ss_tf32(tmem + kColS, dQh + kstep(kk, kQChunk), dKh + kstep(kk, kKChunk), kIdescS,
                      kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < nks; ++kk)
          mma_ss_tf32(tmem + kColS, dQh + kstep(kk, kQChunk), dKl + kstep(kk, kKChunk), kIdescS, 1u);
#pragma unroll
        for (int kk = 0; kk < nks; ++kk)
          mma_ss_tf32(tmem + kColS, dQl + kstep(kk, kQChunk), dKh + kstep(kk, kKChunk), kIdescS, 1u);
        mma_commit(&bars->s_full);
        mma_commit(&bars->k_empty[s]);
      }
      __syncwarp();
    }
    if (!ok && leader) tf32_abort(bars, p.status);
    // no MMA may be in flight when TMEM is released
    mma_commit_w(&bars->drain, leader ? 1u : 0u);
    mbar_wait(&bars->drain, 0, nullptr, kDrainBudget);
    __syncwarp();
  } else if (run && warp >= 2 && warp <= 5) {
    // ======================= softmax / epilogue (warps 2-5) =======================
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
    const int q_row = qt * kBM + row;
    const float c = p.scale_log2;   // any sign: scores are scaled before the max
    float m_ref = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full, j & 1, abort_flag, kWaitBudget))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[kBN];
#pragma unroll
      for (int cc = 0; cc < kBN / 32; ++cc)
        tmem_ld32(tmem + lb + kColS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]));
      tmem_ld_wait(sr);
      tc_fence_before();
      mbar_arrive(&bars->s_free);   // S may take the next block's scores
      float t[kBN];
#pragma unroll
      for (int i = 0; i < kBN; ++i) t[i] = __uint_as_float(sr[i]) * c;
      const int k0 = j * kBN;
      if ((kCausal && k0 + kBN - 1 > qt * kBM) || k0 + kBN > N) {
        const int lim = min(N - 1 - k0, kCausal ? q_row - k0 : kBN - 1);
        // one 32-bit keep mask per 32 columns, a bit select per score
#pragma unroll
        for (int k = 0; k < kBN / 32; ++k) {
          const int sh = lim - 32 * k;   // keep columns 32k .. 32k + sh
          const uint32_t keep =
              sh >= 31 ? 0xffffffffu : (sh < 0 ? 0u : (0xffffffffu >> (31 - sh)));
#pragma unroll
          for (int i = 0; i < 32; ++i) t[32 * k + i] = ((keep >> i) & 1u) ? t[32 * k + i] : -INFINITY;
        }
      }
      float m_blk = -INFINITY;
#pragma unroll
      for (int i = 0; i < kBN; ++i) m_blk = fmaxf(m_blk, t[i]);
      // lazy rescale: move the reference max only when it rises enough
      const bool rise = (m_ref == -INFINITY) ? (m_blk != -INFINITY)
                                             : (m_blk > m_ref + kRescaleThreshold);
      float alpha = 1.0f;
      if (rise) {
        alpha = (m_ref == -INFINITY) ? 0.0f : fast_exp2(m_ref - m_blk);
        m_ref = m_blk;
      }
      l *= alpha;
      const float m_use = (m_ref == -INFINITY) ? 0.0f : m_ref;
      uint32_t ph[kBN], pl[kBN];
      float ls = 0.0f;
#pragma unroll
      for (int i = 0; i < kBN; ++i) {
        const float pv = fast_exp2(t[i] - m_use);
        ls += pv;
        const float hi = tf32_rn(pv);
        ph[i] = __float_as_uint(hi);
        pl[i] = __float_as_uint(tf32_rn(pv - hi));
      }
      l += ls;
      const bool rescale = j > 0 && __any_sync(0xffffffffu, rise);
      // P and O are free once the previous block's PV has completed
      if (j > 0 &&
          !__all_sync(0xffffffffu, mbar_wait(&bars->pv_done, (j - 1) & 1, abort_flag, kWaitBudget))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (rescale) {
#pragma unroll
        for (int cc = 0; cc < kDP / 32; ++cc) {
          uint32_t orr[32];
          __syncwarp();
          tmem_ld32(tmem + lb + kColO + cc * 32, orr);
          tmem_ld_wait(orr);
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
          tmem_st32(tmem + lb + kColO + cc * 32, orr);
        }
      }
      __syncwarp();
#pragma unroll
      for (int cc = 0; cc < kBN / 32; ++cc) {
        tmem_st32(tmem + lb + kColPh + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&ph[cc * 32]));
        tmem_st32(tmem + lb + kColPl + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&pl[cc * 32]));
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }
    if (ok && !__all_sync(0xffffffffu,
                          mbar_wait(&bars->pv_done, (nb - 1) & 1, abort_flag, kWaitBudget)))
      ok = false;
    if (ok) {
      // ---- epilogue: O / l in float32, L = (m + log2 l) ln 2 ----
      tc_fence_after();
      const bool live = l > 0.0f;
      const float inv = live ? 1.0f / l : 0.0f;
      const bool store = q_row < N;
      float* orow = static_cast<float*>(p.o) +
                    ((static_cast<size_t>(b) * N + (store ? q_row : 0)) * H + h) * p.d;
#pragma unroll
      for (int cc = 0; cc < kDP / 32; ++cc) {
        uint32_t orr[32];
        __syncwarp();
        tmem_ld32(tmem + lb + kColO + cc * 32, orr);
        tmem_ld_wait(orr);
        if (store) {
#pragma unroll
          for (int qv = 0; qv < 8; ++qv) {
            const int col = cc * 32 + qv * 4;
            if (col < p.d)
              *reinterpret_cast<float4*>(orow + col) =
                  make_float4(__uint_as_float(orr[qv * 4 + 0]) * inv,
                              __uint_as_float(orr[qv * 4 + 1]) * inv,
                              __uint_as_float(orr[qv * 4 + 2]) * inv,
                              __uint_as_float(orr[qv * 4 + 3]) * inv);
          }
        }
      }
      if (store)
        p.lse[(static_cast<size_t>(b) * H + h) * N + q_row] =
            live ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    } else {
      tf32_abort(bars, p.status);
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
}  // namespace fa

namespace fa {
namespace {

int round4(int n) { return (n + 3) & ~3; }

}  // namespace

// Workspace: Qh, Ql, Kh, Kl ([B, N, H, d] float32 each), V^Th, V^Tl
// ([B, H, d, Np] float32 each), each part rounded up to 256 bytes.
size_t tf32x3_workspace_bytes(int B, int H, int N, int d) {
  const size_t a = (static_cast<size_t>(B) * N * H * d * 4 + 255) & ~static_cast<size_t>(255);
  const size_t t =
      (static_cast<size_t>(B) * H * d * round4(N) * 4 + 255) & ~static_cast<size_t>(255);
  return 4 * a + 2 * t;
}

namespace {

template <int DP>
cudaError_t launch_t3(const FwdParams& p, void* workspace, cudaStream_t st, bool causal) {
  using Cfg = T3Cfg<DP>;
  const int B = p.B, H = p.H, N = p.N, d = p.d, Np = round4(N);
  const size_t a = (static_cast<size_t>(B) * N * H * d * 4 + 255) & ~static_cast<size_t>(255);
  const size_t t = (static_cast<size_t>(B) * H * d * Np * 4 + 255) & ~static_cast<size_t>(255);
  char* w = static_cast<char*>(workspace);
  float *qh = reinterpret_cast<float*>(w), *ql = reinterpret_cast<float*>(w + a),
        *kh = reinterpret_cast<float*>(w + 2 * a), *kl = reinterpret_cast<float*>(w + 3 * a),
        *vth = reinterpret_cast<float*>(w + 4 * a), *vtl = reinterpret_cast<float*>(w + 4 * a + t);
  // tensor maps: [B, N, H, d] as (d, H, N, B); V^T [B, H, d, Np] as (Np, d, H, B)
  const cuuint64_t dq[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                            static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
  const cuuint64_t sq[3] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(H) * d * 4,
                            static_cast<cuuint64_t>(N) * H * d * 4};
  const cuuint64_t dv[4] = {static_cast<cuuint64_t>(Np), static_cast<cuuint64_t>(d),
                            static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t sv[3] = {static_cast<cuuint64_t>(Np) * 4, static_cast<cuuint64_t>(d) * Np * 4,
                            static_cast<cuuint64_t>(H) * d * Np * 4};
  const cuuint32_t box_q[4] = {32u, 1u, static_cast<cuuint32_t>(kBM), 1u};
  const cuuint32_t box_k[4] = {32u, 1u, static_cast<cuuint32_t>(Cfg::kBN), 1u};
  const cuuint32_t box_v[4] = {32u, static_cast<cuuint32_t>(DP), 1u, 1u};
  CUtensorMap mqh, mql, mkh, mkl, mvh, mvl;
  cudaError_t e = make_f32_tmap(&mqh, qh, dq, sq, box_q);
  if (e == cudaSuccess) e = make_f32_tmap(&mql, ql, dq, sq, box_q);
  if (e == cudaSuccess) e = make_f32_tmap(&mkh, kh, dq, sq, box_k);
  if (e == cudaSuccess) e = make_f32_tmap(&mkl, kl, dq, sq, box_k);
  if (e == cudaSuccess) e = make_f32_tmap(&mvh, vth, dv, sv, box_v);
  if (e == cudaSuccess) e = make_f32_tmap(&mvl, vtl, dv, sv, box_v);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return cudaErrorInvalidDevice;
  // Q and K: B N H d is a multiple of 4 (d is a multiple of 8) and the inputs
  // are 16-byte aligned.
  const size_t n4 = static_cast<size_t>(B) * N * H * d / 4;
  const size_t want = (n4 + 255) / 256, cap = static_cast<size_t>(sms) * 8;
  split_qk_kernel<<<static_cast<unsigned>(want < cap ? want : cap), 256, 0, st>>>(
      static_cast<const float4*>(p.q), static_cast<const float4*>(p.k),
      reinterpret_cast<float4*>(qh), reinterpret_cast<float4*>(ql), reinterpret_cast<float4*>(kh),
      reinterpret_cast<float4*>(kl), n4);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (static_cast<long long>(B) * H > 65535) return cudaErrorInvalidConfiguration;
  split_vt_kernel<<<dim3((Np + 31) / 32, (d + 63) / 64, B * H), 256, 0, st>>>(
      static_cast<const float*>(p.v), vth, vtl, N, H, d, Np);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long ctas = static_cast<long long>(B) * H * ((N + kBM - 1) / kBM);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  auto kern = causal ? fwd_tf32x3_kernel<DP, true> : fwd_tf32x3_kernel<DP, false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  FwdParams pc = p;
  void* args[] = {&mqh, &mql, &mkh, &mkl, &mvh, &mvl, &pc};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kern), dim3(static_cast<unsigned>(ctas)),
                          dim3(kThreads), args, Cfg::kSmemBytes, st);
}

}  // namespace

cudaError_t launch_fwd_tf32x3(const FwdParams& p, void* workspace, cudaStream_t st, bool causal) {
  if (p.d % 8 != 0 || p.d > 128) return cudaErrorNotSupported;
  return p.d <= 64 ? launch_t3<64>(p, workspace, st, causal) : launch_t3<128>(p, workspace, st, causal);
}


}  // namespace fa
