// tc_fwd.cu — bf16 fused attention forward on the sm_103a tensor cores.
//
// Algorithm: "Flash Attention 2 — forward pass notes", sections "Loop (per
// (b, h, Q-tile))" and "What's still needed for full FA2" item 1.  FA2 loop
// order: a Q tile stays on chip, K/V blocks stream past it, and each query row
// keeps the online-softmax state (m, l, O) so the N x N scores never reach
// global memory; the per-row log-sum-exp L = m + log l is written at the end.
//
// GB300 mapping: a persistent kernel, one CTA per SM, 12 warps.
//   * Work item = two adjacent 128-row Q tiles (2p, 2p+1) of one (b, h); both
//     read every K/V block the shorter one needs, so each block is loaded once
//     for the pair.  Items are numbered head-major, so the CTAs working at one
//     time share a few heads' K/V through L2; the static round-robin schedule
//     runs odd waves in reverse CTA order, pairing a CTA's short causal items
//     with long ones.
//   * Split-KV mode (kSplit): an item is (tile pair, key slice); the tiles
//     visit only the slice's blocks and write O normalised over the slice and
//     the slice's L, in float32, for a separate merge kernel.
//   * warp 0 (one lane) issues TMA tile loads: K_j and V_j (and with d = 128
//     the item's Q tiles) into a ring of shared-memory stages guarded by full/empty
//     mbarriers.  The ring's position and every barrier's phase carry over
//     from item to item, so the next item's loads overlap this item's tail.
//   * one lane issues the tcgen05 MMAs: S_g = Q_g K_j^T (both operands
//     K-major in smem, fp32 accumulator in TMEM) and O_g += P_g V_j (P read
//     from TMEM, V as an MN-major smem operand).  With d <= 64 warps 1 and 2
//     each issue one tile's MMAs and warp 3 loads Q (two buffers per tile, so
//     the next item's Q lands early); with d = 128 warp 1 interleaves both
//     tiles' MMAs.  Either way one tile's softmax overlaps the other tile's
//     MMAs.
//   * warps 4-7 and 8-11 are the softmax warpgroups of tiles 0 and 1: one
//     thread per query row (= TMEM lane) loads its row of S, masks, takes the
//     row max, exponentiates in base 2 with scale*log2(e) folded in, writes P
//     as 16-bit pairs into TMEM (its own columns with d <= 64, over S's with
//     d = 128), and keeps m and l in registers.
//     O is rescaled by alpha = 2^(m_old - m_new) in TMEM when the running
//     max rises by more than kRescaleThreshold (log2 units, set to 0); warps
//     whose rows' maxima did not move skip the rescale.  After an item's last block each
//     thread divides its O row by l, rounds once to 16 bits and stores it, and
//     stores L in natural-log units; meanwhile the MMA warp already computes
//     the next item's first scores.
//   * the producer/MMA warpgroup gives registers to the softmax warpgroups
//     (setmaxnreg), which hold a full 128-score row per thread.
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

#include <cfloat>
#include <cmath>

#include "fa_common.cuh"
#include "sm103_ptx.cuh"
#include "tmap.h"

namespace fa {
namespace {

constexpr int kBM = 128;                 // query rows per Q tile (= TMEM lanes)
constexpr int kBN = 128;                 // keys per K/V block
constexpr int kQT = 2;                   // Q tiles per work item
constexpr int kThreads = 384;            // 12 warps
constexpr int kChunkBytes = kBM * 128;   // one 64-column swizzled chunk of 128 rows
constexpr int kTmemCols = 512;
// O and l are rescaled whenever a row's running max rises (FWD's alpha rule).
// The reference max is then the exact running max, so the weight of a row's
// largest score is 2^0 = 1, exact in 16 bits: a row dominated by one key gets
// that key's V unperturbed by the rounding of its weight (a threshold of 8,
// i.e. a lazy reference, cost that exactness: weights up to 2^8 rounded to
// 16 bits put up to 2^-9 |V| into O).  Costs ~2 % on the causal GPT-2 shape.
constexpr float kRescaleThreshold = 0.0f;
constexpr int kRegsLoad = 72;            // warps 0-3 (TMA, MMA, Q loads)
constexpr int kRegsSoftmax = 216;        // warps 4-11
// Registers move between warps within an SM sub-partition (warps k, k + 4,
// k + 8: one load/MMA warp and two softmax warps), so the split must fit each
// sub-partition's launch allocation, not only the CTA's.
static_assert(kRegsLoad + 2 * kRegsSoftmax <= 3 * 168 &&
                  4 * 32 * kRegsLoad + 8 * 32 * kRegsSoftmax <= 168 * kThreads,
              "register split exceeds the launch allocation");

// TMEM columns.  S_g: [128 g, 128 g + 128).  O_g: [256 + DP g, 256 + DP g + DP).
// With DP = 64 the 128 columns left over hold P_g (bf16 pairs) at
// [384 + 64 g, 448 + 64 g), so the next S of a tile can be computed while its
// softmax still works on the current block and the previous PV overlaps the
// next softmax.  With DP = 128 TMEM is full and P_g is written over the first
// 64 columns of S_g, so a tile's next S waits until its PV has been issued.
template <int DP>
struct FwdCfg {
  static constexpr bool kSepP = (DP == 64);
  static constexpr int kChunks = DP / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStages = (DP == 64) ? 4 : 2;
  // separate-P layout: two Q buffers per tile slot (the next item's Q loads
  // while this one runs) and a staging tile per slot for the TMA store of O
  static constexpr int kQBufs = kSepP ? 2 : 1;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQT * kQBufs * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kOOff = kVOff + kStages * kTileBytes;
  static constexpr int kBarOff = kOOff + (kSepP ? kQT * kTileBytes : 0);
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;   // + barriers, + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per block");
};

struct FwdBars {
  uint64_t q_full[kQT][2];    // [slot][buffer]; aliased layout: [0][0] for both tiles
  uint64_t q_empty[kQT][2];
  uint64_t k_full[4];
  uint64_t v_full[4];
  uint64_t kv_empty[4];
  uint64_t s_full[kQT];
  uint64_t s_free[kQT];    // softmax has loaded S (separate-P layout)
  uint64_t p_full[kQT];
  uint64_t pv_done[kQT];   // O += P V of a block has completed (separate-P layout)
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

// Bounded wait with a warp-uniform outcome (for roles run by a whole warp).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* ab,
                                          long long budget) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab, budget));
}

// Work item -> (b, h) and its two adjacent Q tiles (2p, 2p+1); with one tile
// (odd tile count, last pair) it is tile[0].  The two tiles' softmax
// warpgroups are both busy for all but the last block, so their MMAs and
// exponentials interleave.
struct Item {
  int b, h;
  int tile[kQT];   // Q tile index, or -1
  int nblk[kQT];   // K blocks each tile visits
  int nmax;
  int j0;          // first K block of the item (split-KV: the slice's first block)
  int split;       // key slice (split-KV), else 0
};

// Split-KV work items of one head, in the causal case.  Pair p (tiles 2p and
// 2p+1) has keys in blocks [0, 2p+2), i.e. ceil((p+1)/hb) slices of 2 hb
// blocks, so the pairs fall into groups k = 1, 2, ... of hb pairs with k slices
// each, and hb (k-1) k / 2 items come before group k.
__host__ __device__ __forceinline__ long long causal_split_items(int npairs, int hb) {
  const long long F = npairs / hb, r = npairs % hb;
  return hb * F * (F + 1) / 2 + r * (F + 1);
}
__device__ __forceinline__ void causal_split_decode(int x, int hb, int& pr, int& sl) {
  int k = static_cast<int>(0.5f * (1.0f + sqrtf(1.0f + 8.0f * static_cast<float>(x) /
                                                        static_cast<float>(hb))));
  k = max(k, 1);
  while (k > 1 && static_cast<long long>(hb) * (k - 1) * k / 2 > x) --k;
  while (static_cast<long long>(hb) * k * (k + 1) / 2 <= x) ++k;
  const int off = x - static_cast<int>(static_cast<long long>(hb) * (k - 1) * k / 2);
  pr = (k - 1) * hb + off / k;
  sl = off % k;
}

// Work items of the whole launch.  Split-KV: one item per (tile pair, key
// slice) that the pair's longer tile reads.
__host__ __device__ __forceinline__ long long fwd_items(int B, int H, int nq, int nk, bool causal,
                                                         bool split, int split_blocks) {
  const int npairs = (nq + 1) / 2;
  long long per_head = npairs;
  if (split)
    per_head = causal ? causal_split_items(npairs, split_blocks / 2)
                      : static_cast<long long>(npairs) * ((nk + split_blocks - 1) / split_blocks);
  return per_head * B * H;
}

template <bool kCausal, bool kSplit>
__device__ __forceinline__ Item decode_item(int it, int nq, int nk, int H, int split_blocks) {
  const int npairs = (nq + 1) / 2;
  Item r;
  int bh, pr, sl = 0;
  if constexpr (!kSplit) {
    bh = it / npairs;
    pr = it % npairs;
  } else if constexpr (kCausal) {
    const int per_head = static_cast<int>(causal_split_items(npairs, split_blocks / 2));
    bh = it / per_head;
    causal_split_decode(it % per_head, split_blocks / 2, pr, sl);
  } else {
    const int ns = (nk + split_blocks - 1) / split_blocks;
    bh = it / (npairs * ns);
    pr = (it / ns) % npairs;
    sl = it % ns;
  }
  r.b = bh / H;
  r.h = bh % H;
  r.split = sl;
  r.j0 = kSplit ? sl * split_blocks : 0;
  const int lo = 2 * pr, hi = 2 * pr + 1;
  r.tile[0] = (hi < nq) ? hi : lo;
  r.tile[1] = (hi < nq) ? lo : -1;
  // Causal: the later tile reads one block more.  Odd items give it to slot
  // 1, so neither slot's lead over the other grows from item to item (the
  // shared K/V ring caps that lead, and a slot at the cap would idle).
  if (kCausal && (it & 1) && r.tile[1] >= 0) {
    r.tile[0] = lo;
    r.tile[1] = hi;
  }
#pragma unroll
  for (int g = 0; g < kQT; ++g) {
    const int all = (r.tile[g] < 0) ? 0 : (kCausal ? min(nk, r.tile[g] + 1) : nk);
    // a slice's blocks [j0, j0 + split_blocks); a tile with none of them is idle
    r.nblk[g] = kSplit ? max(0, min(all, r.j0 + split_blocks) - r.j0) : all;
    if (r.nblk[g] == 0) r.tile[g] = -1;
  }
  r.nmax = max(r.nblk[0], r.nblk[1]);
  return r;
}

// Static schedule: the li-th item of this CTA.  Wave li covers items
// [li*G, (li+1)*G) (G = grid size), so the CTAs working at one time share a
// few heads; odd full waves run in reverse CTA order, which pairs a CTA's
// short causal items with long ones (with G a multiple of the items per head,
// a CTA alternates between complementary tile pairs).  Returns -1 when done.
__device__ __forceinline__ int item_index(int li, int num_items) {
  const long long G = gridDim.x, c = blockIdx.x;
  const long long base = static_cast<long long>(li) * G;
  if (base >= num_items) return -1;
  const bool reverse = (li & 1) && base + G <= num_items;
  const long long it = base + (reverse ? G - 1 - c : c);
  return it < num_items ? static_cast<int>(it) : -1;
}

template <int DP, bool kCausal, bool kF16, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdParams p) {
  using Cfg = FwdCfg<DP>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + Cfg::kBarOff);
  const volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;

  const int N = p.N, H = p.H;
  const int nq = (N + kBM - 1) / kBM;           // Q tiles per head
  const int nk = (N + kBN - 1) / kBN;           // K blocks per head
  const int num_items =
      static_cast<int>(fwd_items(p.B, H, nq, nk, kCausal, kSplit, p.split_blocks));

  // ---- setup: barriers, TMEM ----
  if (threadIdx.x == 0) {
#pragma unroll
    for (int g = 0; g < kQT; ++g) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&bars->q_full[g][b], 1);
        mbar_init(&bars->q_empty[g][b], 1);
      }
      mbar_init(&bars->s_full[g], 1);
      mbar_init(&bars->s_free[g], kBM);
      mbar_init(&bars->p_full[g], kBM);
      mbar_init(&bars->pv_done[g], 1);
      mbar_init(&bars->o_final[g], 1);
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      // separate-P layout: one arrival per softmax warpgroup; else one commit
      mbar_init(&bars->kv_empty[s], Cfg::kSepP ? kQT : 1);
    }
    mbar_init(&bars->drain, Cfg::kSepP ? kQT : 1);   // one commit per MMA warp
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
  uint8_t* sO = smem + Cfg::kOOff;

  // Role bodies; each runs inside the branch that sets its register budget.
  auto load_roles = [&](int warp, int lane) {
    if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int c = 0;             // K/V blocks issued so far
      int li = 0;            // items started by this CTA
      bool ok = true;
      for (int it = item_index(0, num_items); it >= 0 && ok; it = item_index(li, num_items)) {
        const Item w = decode_item<kCausal, kSplit>(it, nq, nk, H, p.split_blocks);
        if constexpr (!Cfg::kSepP) {   // separate-P layout: Q comes from warp 3
          if (li > 0 && !mbar_wait(&bars->q_empty[0][0], (li - 1) & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
          const int nact = (w.tile[1] < 0) ? 1 : 2;
          mbar_arrive_expect_tx(&bars->q_full[0][0], nact * Cfg::kTileBytes);
          for (int g = 0; g < nact; ++g)
            for (int ch = 0; ch < Cfg::kChunks; ++ch)
              tma_load_4d(sQ + g * Cfg::kTileBytes + ch * kChunkBytes, &tmQ, &bars->q_full[0][0],
                          ch * 64, w.h, w.tile[g] * kBM, w.b);
        }
        ++li;
        for (int j = 0; j < w.nmax; ++j) {
          const int s = c % S, round = c / S;
          if (round > 0 &&
              !mbar_wait(&bars->kv_empty[s], (round - 1) & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->k_full[s], Cfg::kTileBytes);
          for (int ch = 0; ch < Cfg::kChunks; ++ch)
            tma_load_4d(sK + s * Cfg::kTileBytes + ch * kChunkBytes, &tmK, &bars->k_full[s],
                        ch * 64, w.h, (w.j0 + j) * kBN, w.b);
          mbar_arrive_expect_tx(&bars->v_full[s], Cfg::kTileBytes);
          for (int ch = 0; ch < Cfg::kChunks; ++ch)
            tma_load_4d(sV + s * Cfg::kTileBytes + ch * kChunkBytes, &tmV, &bars->v_full[s],
                        ch * 64, w.h, (w.j0 + j) * kBN, w.b);
          // Separate-P layout: a tile slot that does not read this block
          // (the shorter causal tile's last block, an absent tile) has its
          // release made here: the stage's previous round is complete, so
          // the arrival counts toward this one.
          if constexpr (Cfg::kSepP)
            for (int g = 0; g < kQT; ++g)
              if (j >= w.nblk[g]) mbar_arrive(&bars->kv_empty[s]);
          ++c;
        }
      }
      if (!ok) raise_abort(bars, p.status);
      // Drain: every issued copy has landed before the CTA may exit.  c counts
      // the K/V blocks issued; the last Q load of each slot is its last phase.
      for (int x = max(0, c - S); x < c; ++x) {
        mbar_wait(&bars->k_full[x % S], (x / S) & 1, nullptr, kDrainBudget);
        mbar_wait(&bars->v_full[x % S], (x / S) & 1, nullptr, kDrainBudget);
      }
      if (!Cfg::kSepP && li > 0)
        mbar_wait(&bars->q_full[0][0], (li - 1) & 1, nullptr, kDrainBudget);
    }
    __syncwarp();
    } else if (Cfg::kSepP && warp == 3) {
    // ============ Q producer (separate-P layout): two buffers per tile slot ============
    if (lane == 0) {
      int li = 0;
      int qn[kQT] = {0, 0};   // Q loads per slot; load n uses buffer n & 1
      bool ok = true;
      for (int it = item_index(0, num_items); it >= 0 && ok; it = item_index(++li, num_items)) {
        const Item w = decode_item<kCausal, kSplit>(it, nq, nk, H, p.split_blocks);
        for (int g = 0; g < kQT; ++g) {
          if (w.tile[g] < 0) continue;
          const int b = qn[g] & 1, u = qn[g] >> 1;
          // the buffer's previous use (load n - 2) has had all its scores computed
          if (u > 0 &&
              !mbar_wait(&bars->q_empty[g][b], (u - 1) & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->q_full[g][b], Cfg::kTileBytes);
          for (int ch = 0; ch < Cfg::kChunks; ++ch)
            tma_load_4d(sQ + (g * 2 + b) * Cfg::kTileBytes + ch * kChunkBytes, &tmQ,
                        &bars->q_full[g][b], ch * 64, w.h, w.tile[g] * kBM, w.b);
          ++qn[g];
        }
      }
      if (!ok) raise_abort(bars, p.status);
      for (int g = 0; g < kQT; ++g)
        for (int n = max(0, qn[g] - 2); n < qn[g]; ++n)
          mbar_wait(&bars->q_full[g][n & 1], (n >> 1) & 1, nullptr, kDrainBudget);
    }
    __syncwarp();
    } else if (warp == 1 || (Cfg::kSepP && warp == 2)) {
    // ================ MMA issuers (whole warp waits, lane 0 issues) ================
    {
      const uint32_t leader = (lane == 0) ? 1u : 0u;
      // A negative scale is applied as a sign flip of Q inside the score MMA
      // (instruction-descriptor bit 13, negate A), so the softmax always
      // works with a positive scale.
      const uint32_t kIdescQK =
          idesc16<kF16>(kBM, kBN, false, false) | (p.scale_log2 < 0.0f ? (1u << 13) : 0u);
      constexpr uint32_t kIdescPV = idesc16<kF16>(kBM, DP, false, true);
      const int nks = (p.d + 15) / 16;       // K=16 steps over the head dim
      // Descriptor bases; K steps and stages advance the start-address field.
      const uint64_t dQ = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(sV), kChunkBytes, 1024);
      auto kstep = [](int kk) -> uint64_t {
        return static_cast<uint64_t>(((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4);
      };
      // scores of tile g from the Q tile at index qi (slot-major, then buffer)
      auto issue_s = [&](int g, int qi, int s) {
        const uint64_t qa = dQ + ((qi * Cfg::kTileBytes) >> 4);
        const uint64_t ka = dK + ((s * Cfg::kTileBytes) >> 4);
        if (leader) {
          // d = DP = 64: fully unrolled, constant offsets, so the single
          // issuing thread spends few instructions per MMA (at DP = 128 the
          // unrolled form costs spills, so the loop stays)
          if (DP == 64 && nks == DP / 16) {
#pragma unroll
            for (int kk = 0; kk < DP / 16; ++kk)
              mma_ss(tmem + g * kBN, qa + kstep(kk), ka + kstep(kk), kIdescQK, kk > 0);
          } else {
            // descriptors advanced in place: +32 B per K=16 step inside a
            // 64-column chunk, then on to the next chunk
            constexpr uint64_t kJump = (kChunkBytes - 96) >> 4;
            uint64_t a = qa, b = ka;
            for (int kk = 0; kk < nks; ++kk) {
              mma_ss(tmem + g * kBN, a, b, kIdescQK, kk > 0);
              const uint64_t inc = (kk & 3) == 3 ? kJump : 2;
              a += inc;
              b += inc;
            }
          }
          mma_commit(&bars->s_full[g]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int g, int s, bool acc) {
        const uint64_t va = dV + ((s * Cfg::kTileBytes) >> 4);
        const uint32_t pa = Cfg::kSepP ? tmem + 384 + g * 64 : tmem + g * kBN;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts(tmem + 2 * kBN + g * DP, pa + kk * 8, va + ((kk * 2048) >> 4), kIdescPV,
                   (acc || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
      };

      int c = 0;                 // K/V blocks consumed so far (same count as the producer)
      int pc[kQT] = {0, 0};      // p_full phases consumed per tile
      int sk[kQT] = {0, 0};      // S MMAs issued per tile (separate-P layout)
      int li = 0;
      bool ok = true;
      if constexpr (Cfg::kSepP) {
        // One MMA warp per Q tile slot (g = warp - 1), so the two tiles never
        // wait on each other's softmax.  Per block j of the tile: S(j) as soon
        // as the softmax has S(j-1) in registers, then O += P(j-1) V(j-1) as
        // soon as P(j-1) is in TMEM.  The sequence runs on across items: the
        // next item's S(0) is issued before this item's last P V (the softmax
        // writes the finished item's O out between its next item's first
        // block and that block's P, so the next P V finds O read).  One
        // commit per MMA group (each costs tensor-pipe time): s_full after S,
        // pv_done after P V; the softmax warpgroup releases K/V stages once
        // it has seen the P V complete.
        const int g = warp - 1;
        int qn = 0;     // Q buffers consumed
        // the P V still to issue: its K/V block index and accumulate flag
        bool pend = false, pend_acc = false, pend_last = false;
        int pend_x = 0;
        auto issue_pending = [&]() -> bool {   // O += P V of the pending block
          const int s = pend_x % S;
          if (!warp_wait(&bars->v_full[s], (pend_x / S) & 1, abort_flag, kWaitBudget) ||
              !warp_wait(&bars->p_full[g], pc[g] & 1, abort_flag, kWaitBudget))
            return false;
          ++pc[g];
          tc_fence_after();
          issue_pv(g, s, pend_acc);
          mma_commit_w(&bars->pv_done[g], leader);
          // an item's last block: this slot's release of its stage, made
          // when the P V has read it (the softmax releases the others)
          if (pend_last) mma_commit_w(&bars->kv_empty[s], leader);
          pend = false;
          return true;
        };
        for (int it = item_index(0, num_items); it >= 0 && ok; it = item_index(++li, num_items)) {
          const Item w = decode_item<kCausal, kSplit>(it, nq, nk, H, p.split_blocks);
          const int nb = w.nblk[g];
          const int qb = qn & 1;   // Q buffer of this item (its load number is qn)
          // The pending P V is the previous item's last.  The softmax's
          // release of that item's last stages waits for it, and the
          // producer may need those releases before this item's first K/V
          // block can land; so it is issued first unless that block is
          // already there (then S(0) goes ahead of it without waiting).
          if (pend && (nb == 0 || !__all_sync(0xffffffffu,
                                             mbar_try_wait(&bars->k_full[c % S], (c / S) & 1))) &&
              !issue_pending()) {
            ok = false;
            break;
          }
          if (nb > 0) {
            if (!warp_wait(&bars->q_full[g][qb], (qn >> 1) & 1, abort_flag, kWaitBudget)) {
              ok = false;
              break;
            }
            ++qn;
          }
          for (int j = 0; j < nb && ok; ++j) {
            const int cj = c + j, s = cj % S;
            if (!warp_wait(&bars->k_full[s], (cj / S) & 1, abort_flag, kWaitBudget) ||
                (sk[g] > 0 &&
                 !warp_wait(&bars->s_free[g], (sk[g] - 1) & 1, abort_flag, kWaitBudget))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(g, g * 2 + qb, s);
            ++sk[g];
            // the tile's last scores are issued: once they complete, the
            // producer may reload this Q buffer
            if (j == nb - 1) mma_commit_w(&bars->q_empty[g][qb], leader);
            if (pend && !issue_pending()) {
              ok = false;
              break;
            }
            pend = true;
            pend_x = cj;
            pend_acc = j > 0;
            pend_last = j == nb - 1;
          }
          if (!ok) break;
          c += w.nmax;
        }
        if (ok && pend && !issue_pending()) ok = false;
      } else {
        for (int it = item_index(0, num_items); it >= 0 && ok; it = item_index(++li, num_items)) {
          const Item w = decode_item<kCausal, kSplit>(it, nq, nk, H, p.split_blocks);
          if (!warp_wait(&bars->q_full[0][0], li & 1, abort_flag, kWaitBudget) ||
              !warp_wait(&bars->k_full[c % S], (c / S) & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int g = 0; g < kQT; ++g)
            if (w.nblk[g] > 0) issue_s(g, g, c % S);
          for (int j = 0; j < w.nmax; ++j) {
            const int cj = c + j, s = cj % S;
            if (!warp_wait(&bars->v_full[s], (cj / S) & 1, abort_flag, kWaitBudget)) {
              ok = false;
              break;
            }
            // Every score MMA of this item has been issued by now: once they
            // complete, the producer may load the next item's Q tiles.
            if (j == w.nmax - 1) mma_commit_w(&bars->q_empty[0][0], leader);
            bool k_next = false;
            for (int g = 0; g < kQT; ++g) {
              if (j >= w.nblk[g]) continue;
              if (!warp_wait(&bars->p_full[g], pc[g] & 1, abort_flag, kWaitBudget)) {
                ok = false;
                break;
              }
              ++pc[g];
              tc_fence_after();
              issue_pv(g, s, j > 0);
              if (j + 1 < w.nblk[g]) {
                if (!k_next) {
                  if (!warp_wait(&bars->k_full[(cj + 1) % S], ((cj + 1) / S) & 1, abort_flag,
                                 kWaitBudget)) {
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                  k_next = true;
                }
                issue_s(g, g, (cj + 1) % S);
              } else {
                mma_commit_w(&bars->o_final[g], leader);
              }
            }
            if (!ok) break;
            mma_commit_w(&bars->kv_empty[s], leader);
          }
          c += w.nmax;
        }

      }
      if (!ok && leader) raise_abort(bars, p.status);
      // Drain: no MMA may be in flight when TMEM is released.
      mma_commit_w(&bars->drain, leader);
      mbar_wait(&bars->drain, 0, nullptr, kDrainBudget);
    }
    __syncwarp();
    }
  };
  auto softmax_role = [&]() {
    // ======================= softmax warpgroups =======================
    const int g = (warp - 4) / 4;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + g * kBN;
    const uint32_t tO = tmem + lane_base + 2 * kBN + g * DP;
    const uint32_t tP = tmem + lane_base + 384 + g * 64;   // separate-P layout only
    // |scale| log2(e): a negative scale reaches the softmax as negated scores
    // (see the score MMA); a zero scale, whose weights are uniform over the
    // unmasked keys, as the smallest positive normal float, which makes every
    // exponent 2^(s c - m) round to 1 while masked keys (-inf) still give 0.
    const float c = p.scale_log2 > 0.0f ? p.scale_log2
                                        : (p.scale_log2 < 0.0f ? -p.scale_log2 : FLT_MIN);
    int sc = 0;    // s_full phases consumed
    int oc = 0;    // epilogues done (o_final phases consumed)
    int kc = 0;    // K/V blocks of the items before this one (separate-P layout)
    bool ok = true;
    // Separate-P layout: this warpgroup's release of the K/V stage of global
    // block x, once its own MMAs no longer read it (every block the tile
    // reads but its item's last; the MMA warp releases that one, the
    // producer the blocks the tile skips).
    auto release_kv = [&](int x) {
      if (row == 0) mbar_arrive(&bars->kv_empty[x % S]);
    };

    // Write an item's output rows: O / l rounded once to 16 bits (split-KV:
    // float32 O over the slice), L = (m + log2 l) ln 2.  Called once the
    // item's last O += P V has completed.
    auto write_out = [&](const Item& ew, int eqt, float em, float el) -> bool {
      const int eq_row = eqt * kBM + row;
      tc_fence_after();
      const bool live = el > 0.0f;
      const float inv = live ? 1.0f / el : 0.0f;
      const bool store = eq_row < N;
      if constexpr (kSplit) {
        // split-KV partial: O normalised over the slice, float32, straight
        // from registers (one 16-byte store per 4 columns of the row)
        float* orow = p.o_part +
                      ((static_cast<size_t>(ew.split) * p.B + ew.b) * N + (store ? eq_row : 0)) *
                          static_cast<size_t>(H) * p.d +
                      static_cast<size_t>(ew.h) * p.d;
#pragma unroll
        for (int cc = 0; cc < DP / 32; ++cc) {
          uint32_t orr[32];
          __syncwarp();   // the stores below are per-thread; tcgen05.ld is collective
          tmem_ld32(tO + cc * 32, orr);
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
      } else if constexpr (Cfg::kSepP) {
        // Each warp stages its 32 bf16 rows of O in shared memory in the TMA
        // box layout (rows of 128 bytes, 16-byte chunk c of row r at chunk
        // c ^ (r & 7)) and its lane 0 stores them with one TMA tensor store
        // (rows >= N and columns >= d are not written): no step waits on
        // another warp.  Lane 0 issued the warp's previous store of this
        // staging tile, so it alone waits for that store to have read it.
        uint8_t* stage = sO + g * Cfg::kTileBytes;
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < DP / 32; ++cc) {
          uint32_t orr[32];
          __syncwarp();   // tcgen05.ld is warp-collective
          tmem_ld32(tO + cc * 32, orr);
          tmem_ld_wait(orr);
#pragma unroll
          for (int qv = 0; qv < 4; ++qv) {
            const int chunk = cc * 4 + qv;   // 16-byte chunk of the row (8 columns)
            uint4 v;
            v.x = pack16x2<kF16>(__uint_as_float(orr[qv * 8 + 0]) * inv,
                              __uint_as_float(orr[qv * 8 + 1]) * inv);
            v.y = pack16x2<kF16>(__uint_as_float(orr[qv * 8 + 2]) * inv,
                              __uint_as_float(orr[qv * 8 + 3]) * inv);
            v.z = pack16x2<kF16>(__uint_as_float(orr[qv * 8 + 4]) * inv,
                              __uint_as_float(orr[qv * 8 + 5]) * inv);
            v.w = pack16x2<kF16>(__uint_as_float(orr[qv * 8 + 6]) * inv,
                              __uint_as_float(orr[qv * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(stage + row * 128 + ((chunk ^ (row & 7)) << 4)) = v;
          }
        }
        fence_proxy_async_smem();   // the TMA engine reads what the threads wrote
        __syncwarp();
        if (lane == 0) {
          tma_store_4d(&tmO, stage + quarter * 32 * 128, 0, ew.h, eqt * kBM + quarter * 32, ew.b);
          bulk_commit_group();
        }
      } else {
        __nv_bfloat16* O = static_cast<__nv_bfloat16*>(p.o);
        uint4* orow = reinterpret_cast<uint4*>(
            O + ((static_cast<size_t>(ew.b) * N + (store ? eq_row : 0)) * H + ew.h) * p.d);
#pragma unroll
        for (int cc = 0; cc < DP / 32; ++cc) {
          uint32_t orr[32];
          __syncwarp();   // the stores below are per-thread; tcgen05.ld is collective
          tmem_ld32(tO + cc * 32, orr);
          tmem_ld_wait(orr);
          if (store) {
#pragma unroll
            for (int qv = 0; qv < 4; ++qv) {
              const int col = cc * 32 + qv * 8;
              if (col < p.d) {
                uint4 v;
                v.x = pack16x2<kF16>(__uint_as_float(orr[qv * 8 + 0]) * inv,
                                  __uint_as_float(orr[qv * 8 + 1]) * inv);
                v.y = pack16x2<kF16>(__uint_as_float(orr[qv * 8 + 2]) * inv,
                                  __uint_as_float(orr[qv * 8 + 3]) * inv);
                v.z = pack16x2<kF16>(__uint_as_float(orr[qv * 8 + 4]) * inv,
                                  __uint_as_float(orr[qv * 8 + 5]) * inv);
                v.w = pack16x2<kF16>(__uint_as_float(orr[qv * 8 + 6]) * inv,
                                  __uint_as_float(orr[qv * 8 + 7]) * inv);
                orow[col / 8] = v;
              }
            }
          }
        }
      }
      tc_fence_before();
      if (store) {
        const float L = live ? (em + __log2f(el)) * 0.69314718055994531f : -INFINITY;
        if constexpr (kSplit)
          p.lse_part[((static_cast<size_t>(ew.split) * p.B + ew.b) * H + ew.h) * N + eq_row] = L;
        else
          p.lse[(static_cast<size_t>(ew.b) * H + ew.h) * N + eq_row] = L;
      }
      return true;
    };
    // Separate-P layout: the item whose output is still to be written
    bool epi_pend = false;
    Item ew{};
    int eqt = 0;
    float em = 0.0f, el = 0.0f;
    // Write out the pending item, after waiting for its last P V unless the
    // caller has.
    auto finish_pending = [&](bool wait_pv) -> bool {
      if (wait_pv && !__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[g], (sc - 1) & 1,
                                                        abort_flag, kWaitBudget)))
        return false;
      ++oc;
      epi_pend = false;
      return write_out(ew, eqt, em, el);
    };
    int li = 0;
    for (int it = item_index(0, num_items); it >= 0 && ok; it = item_index(++li, num_items)) {
      const Item w = decode_item<kCausal, kSplit>(it, nq, nk, H, p.split_blocks);
      const int qt = w.tile[g];
      if (qt < 0) {
        if constexpr (Cfg::kSepP) kc += w.nmax;   // the producer releases its stages
        continue;
      }
      const int q_row = qt * kBM + row;
      float m_ref = -INFINITY;   // reference max of the scaled scores, log2 units
      float l = 0.0f;
      for (int j = 0; j < w.nblk[g]; ++j) {
        // warp-uniform outcome: the TMEM accesses below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[g], sc & 1, abort_flag,
                                               kWaitBudget))) {
          ok = false;
          break;
        }
        ++sc;
        tc_fence_after();
        uint32_t sr[kBN];
        tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
        tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
        tmem_ld_wait(sr);
        // a float copy (registers): writing floats through a pointer into the
        // uint32 array would break type-based aliasing rules
        float s[kBN];
#pragma unroll
        for (int i = 0; i < kBN; ++i) s[i] = __uint_as_float(sr[i]);
        if constexpr (Cfg::kSepP) {
          // S is in registers: its TMEM columns may take the next block's S
          tc_fence_before();
          mbar_arrive(&bars->s_free[g]);
        }

        // Blocks with masked keys (the diagonal block of a causal tile, the
        // ragged last block) set them to -inf before the row max: key k0 + i
        // is masked when i > lim (beyond N, or after q_row).  The limit
        // becomes one 32-bit keep mask per 32 columns, and each score a
        // select on one bit of it (cheaper than a compare per score).  One
        // copy of the row loops serves every block (the instruction cache
        // holds it once).
        const int jb = w.j0 + j;   // the block's index among the head's keys
        if ((kCausal && jb == qt) || ((jb + 1) * kBN > N)) {
          const int k0 = jb * kBN;
          const int lim = min(N - k0 - 1, kCausal ? q_row - k0 : kBN);
#pragma unroll
          for (int k = 0; k < kBN / 32; ++k) {
            const int sh = lim - 32 * k;   // keep columns 32k .. 32k + sh
            const uint32_t keep =
                sh >= 31 ? 0xffffffffu : (sh < 0 ? 0u : (0xffffffffu >> (31 - sh)));
#pragma unroll
            for (int i = 0; i < 32; ++i)
              s[32 * k + i] = ((keep >> i) & 1u) ? s[32 * k + i] : -INFINITY;
          }
        }
        bool rise = false;
        float alpha = 1.0f;
        uint32_t pk[kBN / 2];
        {
          float m_blk;
          {
            float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
            for (int i = 0; i < kBN; i += 8) {   // four chains, columns 0 .. kBN-1
              a0 = fmax3(a0, s[i], s[i + 1]);
              a1 = fmax3(a1, s[i + 2], s[i + 3]);
              a2 = fmax3(a2, s[i + 4], s[i + 5]);
              a3 = fmax3(a3, s[i + 6], s[i + 7]);
            }
            m_blk = fmax3(a0, a1, fmaxf(a2, a3)) * c;
          }
          // Move the reference max whenever the row max rises.
          rise = (m_ref == -INFINITY) ? (m_blk != -INFINITY)
                                      : (m_blk > m_ref + kRescaleThreshold);
          if (rise) {
            alpha = (m_ref == -INFINITY) ? 0.0f : fast_exp2(m_ref - m_blk);
            m_ref = m_blk;
          }
          l *= alpha;
          const float m_use = (m_ref == -INFINITY) ? 0.0f : m_ref;
          const uint64_t negm2 = f2_pack(-m_use, -m_use);
          const uint64_t c2 = f2_pack(c, c);
          // P = 2^(s c - m) as bf16 pairs.
          uint64_t lsum0 = 0, lsum1 = 0;   // two packed partial sums (+0.0f pairs)
#pragma unroll
          for (int i = 0; i < kBN / 2; ++i) {
            const uint64_t sv = f2_pack(s[2 * i], s[2 * i + 1]);
            const uint64_t t = f2_fma(sv, c2, negm2);
            const float p0 = fast_exp2(f2_lo(t));
            const float p1 = fast_exp2(f2_hi(t));
            const uint64_t pp = f2_pack(p0, p1);
            if (i & 1) lsum1 = f2_add(lsum1, pp); else lsum0 = f2_add(lsum0, pp);
            pk[i] = pack16x2<kF16>(p0, p1);
          }
          const uint64_t ls = f2_add(lsum0, lsum1);
          l += f2_lo(ls) + f2_hi(ls);
        }
        const bool rescale = j > 0 && __any_sync(0xffffffffu, rise);
        // O row *= alpha in TMEM (warp-collective; alpha is 1 in rows whose
        // max did not move).  Called once O holds every block before this one.
        auto rescale_o = [&]() {
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int cc = 0; cc < DP / 32; ++cc) {
            uint32_t orr[32];
            __syncwarp();   // tcgen05.ld/st are warp-collective
            tmem_ld32(tO + cc * 32, orr);
            tmem_ld_wait(orr);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const uint64_t v = f2_mul(f2_pack(__uint_as_float(orr[i]),
                                                __uint_as_float(orr[i + 1])), a2);
              orr[i] = __float_as_uint(f2_lo(v));
              orr[i + 1] = __float_as_uint(f2_hi(v));
            }
            tmem_st32(tO + cc * 32, orr);
          }
        };
        // Aliased layout: PV of block j-1 has completed, since the s_full
        // commit of block j came after it.
        if (!Cfg::kSepP && rescale) rescale_o();
        if constexpr (Cfg::kSepP) {
          // P_g and O_g are free once PV of the previous block has completed
          // (the pv_done phase of that block; blocks counted across items).
          if (sc >= 2 &&
              !__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[g], sc & 1, abort_flag,
                                                 kWaitBudget))) {
            ok = false;
            break;
          }
          // block j-1's MMAs are done (the previous item's last block is
          // released with its deferred epilogue, here at j = 0)
          if (j > 0) release_kv(kc + j - 1);
          if (j == 0 && epi_pend && !finish_pending(false)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (rescale) rescale_o();
          __syncwarp();
          tmem_st32(tP + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        } else {
          __syncwarp();
          tmem_st32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_full[g]);
      }
      if (!ok) break;

      if constexpr (Cfg::kSepP) {
        // The epilogue is deferred: it runs during the next item's first
        // block, between that block's exponentials and its P store, by when
        // this item's last P V has long completed.
        epi_pend = true;
        ew = w;
        eqt = qt;
        em = m_ref;
        el = l;
        kc += w.nmax;
      } else {
        // ---- epilogue (aliased layout) ----
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&bars->o_final[g], oc & 1, abort_flag, kWaitBudget))) {
          ok = false;
          break;
        }
        ++oc;
        if (!write_out(w, qt, m_ref, l)) {
          ok = false;
          break;
        }
      }
    }
    if (ok && epi_pend) ok = finish_pending(true);
    if (!ok) raise_abort(bars, p.status);
    // the O stores must have completed (and read shared memory) before exit
    if (Cfg::kSepP && lane == 0) bulk_wait_all();
    __syncwarp();
  };

  if (warp < 4) {
    regs_dec<kRegsLoad>();
    if (run) load_roles(warp, lane);
  } else {
    regs_inc<kRegsSoftmax>();
    if (run) softmax_role();
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int DP, bool kCausal, bool kF16, bool kSplit>
cudaError_t launch_tc(const FwdParams& p, cudaStream_t st) {
  using Cfg = FwdCfg<DP>;
  CUtensorMap mq, mk, mv, mo;
  cudaError_t e = make_bhnd_tmap(&mq, p.q, p.B, p.N, p.H, p.d, kBM, 64, kF16);
  if (e == cudaSuccess) e = make_bhnd_tmap(&mk, p.k, p.B, p.N, p.H, p.d, kBM, 64, kF16);
  if (e == cudaSuccess) e = make_bhnd_tmap(&mv, p.v, p.B, p.N, p.H, p.d, kBM, 64, kF16);
  // the split-KV partial pass writes float32 rows directly; its O map is unused
  if (e == cudaSuccess)
    e = make_bhnd_tmap(&mo, kSplit ? p.q : p.o, p.B, p.N, p.H, p.d, 32, 64, kF16);
  if (e != cudaSuccess) return e;
  auto kern = fwd_tc_kernel<DP, kCausal, kF16, kSplit>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int nq = (p.N + kBM - 1) / kBM;
  const int nk = (p.N + kBN - 1) / kBN;
  if (kSplit && (p.split_blocks < 2 || p.split_blocks % 2 != 0)) return cudaErrorInvalidValue;
  const long long items = fwd_items(p.B, p.H, nq, nk, kCausal, kSplit, p.split_blocks);
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  FwdParams pc = p;
  void* args[] = {&mq, &mk, &mv, &mo, &pc};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(kThreads), args,
                          Cfg::kSmemBytes, st);
}

template <bool kF16, bool kSplit>
cudaError_t launch_dtype(const FwdParams& p, cudaStream_t s, bool causal) {
  if (p.d <= 64)
    return causal ? launch_tc<64, true, kF16, kSplit>(p, s)
                  : launch_tc<64, false, kF16, kSplit>(p, s);
  if (p.d <= 128)
    return causal ? launch_tc<128, true, kF16, kSplit>(p, s)
                  : launch_tc<128, false, kF16, kSplit>(p, s);
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_fwd_tc16(const FwdParams& p, cudaStream_t s, bool causal) {
  return p.f16 ? launch_dtype<true, false>(p, s, causal) : launch_dtype<false, false>(p, s, causal);
}

cudaError_t launch_fwd_tc16_partial(const FwdParams& p, cudaStream_t s, bool causal) {
  return p.f16 ? launch_dtype<true, true>(p, s, causal) : launch_dtype<false, true>(p, s, causal);
}

}  // namespace fa
