// tc_fwd.cu — bf16 fused attention forward on the sm_103a tensor cores.
//
// Algorithm: "Flash Attention 2 — forward pass notes", sections "Loop (per
// (b, h, Q-tile))" and "What's still needed for full FA2" item 1.  FA2 loop
// order: a Q tile stays on chip, K/V blocks stream past it, and each query row
// keeps the online-softmax state (m, l, O) so the N x N scores never reach
// global memory; the per-row log-sum-exp L = m + log l is written at the end.
//
// GB300 mapping (one CTA per SM, 12 warps):
//   * a CTA owns two adjacent 128-row Q tiles of one (b, h); both tiles share
//     every K/V block it loads, which halves K/V traffic into shared memory;
//   * warp 0 (one lane) issues TMA tile loads: Q once, then K_j and V_j into a
//     ring of shared-memory stages guarded by full/empty mbarriers;
//   * warp 1 (one lane) issues tcgen05 MMAs: S_g = Q_g K_j^T (both operands
//     K-major in smem, fp32 accumulator in TMEM) and O_g += P_g V_j (P read
//     from TMEM, V as an MN-major smem operand).  MMAs of the two Q tiles
//     interleave so one tile's softmax overlaps the other tile's MMAs;
//   * warps 4-7 and 8-11 are the softmax warpgroups of Q tiles 0 and 1: one
//     thread per query row (= TMEM lane) loads its row of S, masks, takes the
//     row max, exponentiates in base 2 with scale*log2(e) folded in, writes P
//     as bf16 back into the same TMEM columns, and keeps m and l in registers.
//     The output is rescaled by alpha = 2^(m_old - m_new) in TMEM only when the
//     running max rises by more than kRescaleThreshold (log2 units); a stale
//     reference max cancels exactly in O / l and in L.
//   * after the last block each softmax thread divides its O row by l, rounds
//     once to bf16 and stores it, and stores L in natural-log units.
//
// Tiles are stored in shared memory as 64-column (128-byte) chunks with the
// 128-byte swizzle; head dims below the padded width DP are zero-filled by
// TMA's out-of-bounds fill and cost nothing in the result.  Keys >= N (zero
// rows from the same fill) and keys above the diagonal are masked to -inf.
//
// Every mbarrier wait is bounded; a wait that gives up records FA_ERR_TIMEOUT
// in the status word, raises a CTA-wide abort flag, and the CTA drains its
// in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "fa_common.cuh"
#include "sm103_ptx.cuh"
#include "tmap.h"

namespace fa {
namespace {

constexpr int kBM = 128;                 // query rows per Q tile (= TMEM lanes)
constexpr int kBN = 128;                 // keys per K/V block
constexpr int kQT = 2;                   // Q tiles per CTA
constexpr int kThreads = 384;            // 12 warps
constexpr int kChunkBytes = kBM * 128;   // one 64-column swizzled chunk of 128 rows
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;

template <int DP>
struct FwdCfg {
  static constexpr int kChunks = DP / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStages = (DP == 64) ? 4 : 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQT * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;   // + barriers, + alignment slack
};

struct FwdBars {
  uint64_t q_full[kQT];
  uint64_t k_full[4];
  uint64_t v_full[4];
  uint64_t kv_empty[4];
  uint64_t s_full[kQT];
  uint64_t p_full[kQT];
  uint64_t o_final[kQT];
  uint64_t drain;
  uint64_t probe;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void raise_abort(FwdBars* bars, int* status) {
  record_error(status, FA_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&bars->abort) = 1;
}

template <int DP, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using Cfg = FwdCfg<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + Cfg::kBarOff);
  const volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;

  // ---- work item: two adjacent Q tiles of one (b, h); longest rows first ----
  const int N = p.N, H = p.H;
  const int nq = (N + kBM - 1) / kBM;           // Q tiles per head
  const int nk = (N + kBN - 1) / kBN;           // K blocks per head
  const int nqp = (nq + kQT - 1) / kQT;         // Q-tile pairs per head
  // Head-major order: the CTAs of one head run side by side and share its K/V
  // through L2; within a head the longest (causal) tile pair goes first.
  const int item = blockIdx.x;
  const int qp = nqp - 1 - item % nqp;
  const int bh = item / nqp, b = bh / H, h = bh % H;
  const int qt0 = qp * kQT;
  const int n_active = min(kQT, nq - qt0);
  int nblk[kQT];
#pragma unroll
  for (int g = 0; g < kQT; ++g)
    nblk[g] = (g < n_active) ? (kCausal ? min(nk, qt0 + g + 1) : nk) : 0;
  const int nmax = max(nblk[0], nblk[1]);

  // ---- setup: barriers, TMEM ----
  if (threadIdx.x == 0) {
#pragma unroll
    for (int g = 0; g < kQT; ++g) {
      mbar_init(&bars->q_full[g], 1);
      mbar_init(&bars->s_full[g], 1);
      mbar_init(&bars->p_full[g], kBM);
      mbar_init(&bars->o_final[g], 1);
    }
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->drain, 1);
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
    // Self-test of the bounded-wait path: nothing ever arrives on `probe`.
    if (threadIdx.x == 0 && !mbar_wait(&bars->probe, 0, abort_flag, kProbeBudget))
      raise_abort(bars, p.status);
    __syncthreads();
    run = false;
  }

  uint8_t* sQ = smem + Cfg::kQOff;
  uint8_t* sK = smem + Cfg::kKOff;
  uint8_t* sV = smem + Cfg::kVOff;

  if (run && warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      for (int g = 0; g < n_active; ++g) {
        mbar_arrive_expect_tx(&bars->q_full[g], Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_4d(sQ + g * Cfg::kTileBytes + c * kChunkBytes, &tmQ, &bars->q_full[g], c * 64,
                      h, (qt0 + g) * kBM, b);
      }
      int issued = 0;
      for (int j = 0; j < nmax; ++j) {
        const int s = j % Cfg::kStages, round = j / Cfg::kStages;
        if (round > 0 && !mbar_wait(&bars->kv_empty[s], (round - 1) & 1, abort_flag, kWaitBudget)) {
          raise_abort(bars, p.status);
          break;
        }
        mbar_arrive_expect_tx(&bars->k_full[s], Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_4d(sK + s * Cfg::kTileBytes + c * kChunkBytes, &tmK, &bars->k_full[s], c * 64, h,
                      j * kBN, b);
        mbar_arrive_expect_tx(&bars->v_full[s], Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_4d(sV + s * Cfg::kTileBytes + c * kChunkBytes, &tmV, &bars->v_full[s], c * 64, h,
                      j * kBN, b);
        issued = j + 1;
      }
      // Drain: every issued copy has landed before the CTA may exit.
      for (int j = max(0, issued - Cfg::kStages); j < issued; ++j) {
        const int s = j % Cfg::kStages, par = (j / Cfg::kStages) & 1;
        mbar_wait(&bars->k_full[s], par, nullptr, kDrainBudget);
        mbar_wait(&bars->v_full[s], par, nullptr, kDrainBudget);
      }
      for (int g = 0; g < n_active; ++g) mbar_wait(&bars->q_full[g], 0, nullptr, kDrainBudget);
    }
    __syncwarp();
  } else if (run && warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(kBM, DP, false, true);
      const int nks = (p.d + 15) / 16;       // K=16 steps over the head dim
      const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
      bool ok = true;

      auto issue_s = [&](int g, int j) {
        const int s = j % Cfg::kStages;
        const uint32_t qa = sQa + g * Cfg::kTileBytes;
        const uint32_t ka = sKa + s * Cfg::kTileBytes;
        for (int kk = 0; kk < nks; ++kk) {
          const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + g * kBN, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                 kIdescQK, kk > 0);
        }
        mma_commit(&bars->s_full[g]);
      };
      auto issue_pv = [&](int g, int j) {
        const int s = j % Cfg::kStages;
        const uint32_t va = sVa + s * Cfg::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(tmem + 2 * kBN + g * DP, tmem + g * kBN + kk * 8,
                 sdesc_sw128(va + kk * 2048, kChunkBytes, 1024), kIdescPV, (j > 0 || kk > 0));
      };

      for (int g = 0; g < n_active && ok; ++g)
        if (!mbar_wait(&bars->q_full[g], 0, abort_flag, kWaitBudget)) ok = false;
      if (ok && !mbar_wait(&bars->k_full[0], 0, abort_flag, kWaitBudget)) ok = false;
      if (ok) {
        tc_fence_after();
        for (int g = 0; g < n_active; ++g) issue_s(g, 0);
      }
      for (int j = 0; j < nmax && ok; ++j) {
        const int s = j % Cfg::kStages;
        if (!mbar_wait(&bars->v_full[s], (j / Cfg::kStages) & 1, abort_flag, kWaitBudget)) {
          ok = false;
          break;
        }
        bool k_next = false;
        for (int g = 0; g < kQT; ++g) {
          if (j >= nblk[g]) continue;
          if (!mbar_wait(&bars->p_full[g], j & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(g, j);
          if (j + 1 < nblk[g]) {
            if (!k_next) {
              const int s1 = (j + 1) % Cfg::kStages;
              if (!mbar_wait(&bars->k_full[s1], ((j + 1) / Cfg::kStages) & 1, abort_flag,
                             kWaitBudget)) {
                ok = false;
                break;
              }
              tc_fence_after();
              k_next = true;
            }
            issue_s(g, j + 1);
          } else {
            mma_commit(&bars->o_final[g]);
          }
        }
        if (!ok) break;
        mma_commit(&bars->kv_empty[s]);
      }
      if (!ok) raise_abort(bars, p.status);
      // Drain: no MMA may be in flight when TMEM is released.
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, nullptr, kDrainBudget);
    }
    __syncwarp();
  } else if (run && warp >= 4) {
    // ======================= softmax warpgroups =======================
    const int g = (warp - 4) / 4;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int qt = qt0 + g;
    const int q_row = qt * kBM + row;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + g * kBN;
    const uint32_t tO = tmem + lane_base + 2 * kBN + g * DP;
    const float c = p.scale_log2;
    float m_ref = -INFINITY;   // reference max of the scaled scores, log2 units
    float l = 0.0f;
    bool ok = true;

    if (g < n_active) {
      for (int j = 0; j < nblk[g]; ++j) {
        // warp-uniform outcome: the TMEM accesses below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[g], j & 1, abort_flag, kWaitBudget))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[kBN];
        tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
        tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
        tmem_ld_wait(sr);
        float* s = reinterpret_cast<float*>(sr);

        const bool masked = (kCausal && j == qt) || ((j + 1) * kBN > N);
        float m_blk;
        if (masked) {
          const int k0 = j * kBN;
          float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
          for (int i = 0; i < kBN; ++i) {
            const int key = k0 + i;
            const bool bad = (key >= N) || (kCausal && key > q_row);
            s[i] = bad ? -INFINITY : s[i] * c;
            if (i & 1) mx1 = fmaxf(mx1, s[i]); else mx0 = fmaxf(mx0, s[i]);
          }
          m_blk = fmaxf(mx0, mx1);
        } else {
          float a0 = s[0], a1 = s[1], a2 = s[2], a3 = s[3];
          if (c >= 0.0f) {
#pragma unroll
            for (int i = 4; i < kBN; i += 4) {
              a0 = fmaxf(a0, s[i]); a1 = fmaxf(a1, s[i + 1]);
              a2 = fmaxf(a2, s[i + 2]); a3 = fmaxf(a3, s[i + 3]);
            }
            m_blk = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * c;
          } else {
#pragma unroll
            for (int i = 4; i < kBN; i += 4) {
              a0 = fminf(a0, s[i]); a1 = fminf(a1, s[i + 1]);
              a2 = fminf(a2, s[i + 2]); a3 = fminf(a3, s[i + 3]);
            }
            m_blk = fminf(fminf(a0, a1), fminf(a2, a3)) * c;
          }
        }

        // Lazy rescale: move the reference max only when it rises enough.
        const bool rise = (m_ref == -INFINITY) ? (m_blk != -INFINITY)
                                               : (m_blk > m_ref + kRescaleThreshold);
        float alpha = 1.0f;
        if (rise) {
          alpha = (m_ref == -INFINITY) ? 0.0f : fast_exp2(m_ref - m_blk);
          m_ref = m_blk;
        }
        if (j > 0 && __any_sync(0xffffffffu, rise)) {
          // O row *= alpha in TMEM (PV of block j-1 has completed: s_full of
          // block j was committed after it).
#pragma unroll
          for (int cc = 0; cc < DP / 32; ++cc) {
            uint32_t orr[32];
            tmem_ld32(tO + cc * 32, orr);
            tmem_ld_wait(orr);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            tmem_st32(tO + cc * 32, orr);
          }
        }
        l *= alpha;
        const float m_use = (m_ref == -INFINITY) ? 0.0f : m_ref;

        // P = 2^(s c - m) -> bf16 pairs into TMEM columns [0, 64) of S.
        float l0 = 0.0f, l1 = 0.0f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int e = half * 64 + 2 * i;
            float p0, p1;
            if (masked) {
              p0 = fast_exp2(s[e] - m_use);
              p1 = fast_exp2(s[e + 1] - m_use);
            } else {
              p0 = fast_exp2(fmaf(s[e], c, -m_use));
              p1 = fast_exp2(fmaf(s[e + 1], c, -m_use));
            }
            l0 += p0;
            l1 += p1;
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st32(tS + half * 32, pk);
        }
        l += l0 + l1;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_full[g]);
      }

      // ---- epilogue: O / l -> bf16, L = (m + log2 l) ln 2 ----
      if (ok && !__all_sync(0xffffffffu, mbar_wait(&bars->o_final[g], 0, abort_flag, kWaitBudget)))
        ok = false;
      if (ok) {
        tc_fence_after();
        const bool live = l > 0.0f;
        const float inv = live ? 1.0f / l : 0.0f;
        const bool store = q_row < N;
        __nv_bfloat16* O = static_cast<__nv_bfloat16*>(p.o);
        uint4* orow = reinterpret_cast<uint4*>(
            O + ((static_cast<size_t>(b) * N + (store ? q_row : 0)) * H + h) * p.d);
#pragma unroll
        for (int cc = 0; cc < DP / 32; ++cc) {
          uint32_t orr[32];
          tmem_ld32(tO + cc * 32, orr);
          tmem_ld_wait(orr);
          if (store) {
#pragma unroll
            for (int qv = 0; qv < 4; ++qv) {
              const int col = cc * 32 + qv * 8;
              if (col < p.d) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(orr[qv * 8 + 0]) * inv,
                                  __uint_as_float(orr[qv * 8 + 1]) * inv);
                v.y = pack_bf16x2(__uint_as_float(orr[qv * 8 + 2]) * inv,
                                  __uint_as_float(orr[qv * 8 + 3]) * inv);
                v.z = pack_bf16x2(__uint_as_float(orr[qv * 8 + 4]) * inv,
                                  __uint_as_float(orr[qv * 8 + 5]) * inv);
                v.w = pack_bf16x2(__uint_as_float(orr[qv * 8 + 6]) * inv,
                                  __uint_as_float(orr[qv * 8 + 7]) * inv);
                orow[col / 8] = v;
              }
            }
          }
        }
        if (store)
          p.lse[static_cast<size_t>(bh) * N + q_row] =
              live ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
      if (!ok) raise_abort(bars, p.status);
    }
    __syncwarp();
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int DP, bool kCausal>
cudaError_t launch_tc(const FwdParams& p, cudaStream_t st) {
  using Cfg = FwdCfg<DP>;
  CUtensorMap mq, mk, mv;
  cudaError_t e = make_bhnd_tmap(&mq, p.q, p.B, p.N, p.H, p.d);
  if (e == cudaSuccess) e = make_bhnd_tmap(&mk, p.k, p.B, p.N, p.H, p.d);
  if (e == cudaSuccess) e = make_bhnd_tmap(&mv, p.v, p.B, p.N, p.H, p.d);
  if (e != cudaSuccess) return e;
  auto kern = fwd_tc_kernel<DP, kCausal>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int nq = (p.N + kBM - 1) / kBM;
  const long long items = static_cast<long long>((nq + kQT - 1) / kQT) * p.B * p.H;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  FwdParams pc = p;
  void* args[] = {&mq, &mk, &mv, &pc};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kern), dim3(static_cast<unsigned>(items)),
                          dim3(kThreads), args, Cfg::kSmemBytes, st);
}

}  // namespace

cudaError_t launch_fwd_tc_bf16(const FwdParams& p, cudaStream_t s, bool causal) {
  if (p.d <= 64) return causal ? launch_tc<64, true>(p, s) : launch_tc<64, false>(p, s);
  if (p.d <= 128) return causal ? launch_tc<128, true>(p, s) : launch_tc<128, false>(p, s);
  return cudaErrorNotSupported;
}

}  // namespace fa
