// tc_bwd.cu — bf16 attention backward on the sm_103a tensor cores.
//
// Algorithm: "Flash Attention 2 — backward pass notes", section "The math (FA2
// backward with recompute)": with the saved L, P = exp(S - L) is recomputed;
// dP = dO V^T, dS = P (dP - D) with D = <dO, O>, dV = P^T dO,
// dK = scale dS^T Q, dQ = scale dS K.  Split as the same page's option 3 ("Why
// the WGSL kernel isn't shipped this turn"): one kernel whose CTA owns a tile
// of queries and accumulates dQ, one whose CTA owns a tile of keys and
// accumulates dK and dV.  Each output row is written once, by one CTA: no
// float atomics.  Rows whose L is -inf contribute nothing ("Caveats specific
// to the backward path").
//
// Precision.  The forward stores O in bf16, and D computed from that O is off
// by up to |dO| |O| 2^-9 per row; the gradient amplifies that by |K| scale,
// which exceeds the bf16 gradient tolerance when Q and K have large entries.
// The dQ kernel therefore also accumulates the exact-form D_i =
// sum_j P_ij dP_ij in fp32 and B_i = sum_j P_ij K_j, runs its loop with the
// estimate D~ from the bf16 O (formed by the dQ kernel itself from the O and
// dO rows it loads in the wide layout, by the pre-pass bwd_dot.cu in the
// narrow one) and adds scale (D~_i - D_i) B_i at the end
// (algebraically the same dQ); it writes the refined D back to the workspace,
// and the dK/dV kernel, launched after it, uses that.  dS (and P for B) are
// staged for the tensor cores in fp16, whose 11-bit significand keeps the
// product error ~8x below bf16's; the streamed K or Q tile they multiply is
// converted to an fp16 copy in shared memory (an MMA takes one input type).
// This bounds |Q|, |K| and |dS| by fp16's range (65504) in the backward.
//
// Both kernels share one persistent skeleton (template parameter kDkDv): one
// CTA per SM walks work items, each a 128-row tile of one (b, h):
//   row tile   : resident in shared memory for the item.  dQ kernel: Q and dO
//                of 128 queries (and, wide layout, O for D's estimate).
//                dK/dV kernel: K and V of 128 keys.
//   blocks     : streamed through a TMA ring.  dQ: K_j, V_j.  dK/dV: Q_i, dO_i
//                (plus their L and D).
//   per block  : S = R1 C1^T and dP = R2 C2^T (tcgen05, M=128, bf16, both
//                operands K-major); one thread per row forms P and dS and
//                writes them to TMEM; then
//                dQ kernel:    dQ += dS K_j, B += P K_j      (fp16)
//                dK/dV kernel: dV += P dO_i (bf16), dK += dS Q_i (fp16)
//                with A read from TMEM and B the streamed tile as an MN-major
//                operand.
// Two layouts (TMEM is 512 columns):
//   head dim <= 64 ("wide"): 128-row blocks, so the S and dP MMAs are
//     128 x 128; both element-wise warpgroups work on every block (64 columns
//     each); S and dP are released as soon as they are in registers and P, dS
//     have their own columns, so the next block's S and dP MMAs run while the
//     current block's exponentials are computed.
//     columns: S [0,128) dP [128,256) acc1 [256,320) acc2 [320,384)
//              P [384,448) dS [448,512)
//   head dim <= 128 ("narrow"): 64-row blocks; S and dP double-buffered, P and
//     dS written over them, the two warpgroups take alternate blocks.
//     columns: S [0,128) dP [128,256) acc1 [256,384) acc2 [384,512)
// Items are numbered head-major (CTAs working at one time share a few heads'
// streamed tiles through L2) and odd waves run in reverse CTA order, which
// pairs long and short causal tiles on each CTA.
//
// Roles (12 warps): warp 0 TMA producer; warp 1 issues the MMAs (converged,
// lane 0 issues) — in the wide dQ kernels and the wide causal dK/dV kernel
// only S/dP, with warp 3 issuing the first accumulation and warp 2 the second
// (elsewhere warp 1 also issues the first and warp 2 the second); the
// per-query -L2 and -D of each streamed block (dK/dV kernel) are written by
// warp 2 (narrow layout, and one block ahead of its dK MMAs in the wide
// causal kernel) or warp 3 (wide non-causal); the fp16 copy of each streamed
// C1 tile is made by the element-wise warps in the wide layout (in place over
// the bf16 tile, once the block's S has read it) and by warp 3 in the narrow
// one; warps 4-7 and 8-11 are the element-wise warpgroups and the epilogue
// (each stores half of the columns of the accumulator rows; in the wide dK/dV
// kernel an item's epilogue runs during the next item's first block).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "fa_common.cuh"
#include "sm103_ptx.cuh"
#include "tmap.h"

namespace fa {
namespace {

constexpr int kRows = 128;       // rows owned by a work item
constexpr int kThreads = 384;
constexpr int kRegsHelper = 88;    // warps 0-3: TMA, MMA, vectors, fp16 copy
constexpr int kRegsElem = 208;     // warps 4-11: element-wise and epilogue
// Registers move between warps within an SM sub-partition (warps k, k + 4,
// k + 8: one helper and two element-wise warps), so the split must fit each
// sub-partition's launch allocation, not only the CTA's.
static_assert(kRegsHelper + 2 * kRegsElem <= 3 * 168 &&
                  4 * 32 * kRegsHelper + 8 * 32 * kRegsElem <= 168 * kThreads,
              "register split exceeds the launch allocation");
constexpr int kTmemCols = 512;
constexpr int kStagesMax = 4;
constexpr float kLog2e = 1.4426950408889634f;

template <int DP, bool kDkDv>
struct BwdCfg {
  static constexpr bool kWide = (DP == 64);
  // the wide dQ kernel also loads each item's O rows (third row tile): it
  // forms the first estimate of D = rowsum(dO * O) itself, so that path has
  // no D pre-pass
  static constexpr bool kOwnD = kWide && !kDkDv;
  static constexpr int kRTiles = kOwnD ? 3 : 2;
  static constexpr int kBlk = kWide ? 128 : 64;          // rows of one streamed block
  // wide layout: the fp16 copy of C1 overwrites the bf16 tile in place (made
  // once the block's S has been computed, its only bf16 reader), so a stage
  // is two tiles and four stages fit; narrow: a separate copy, three stages
  static constexpr int kStages = 3;
  // wide dK/dV kernel: an item's epilogue is deferred to the next item's first
  // block, so its row buffer (where the gradient rows are staged) is held a
  // little longer; a third buffer keeps the next-but-one item's rows loading
  static constexpr bool kDefer = kWide && kDkDv;
  static constexpr int kChunks = DP / 64;
  static constexpr int kRowChunk = kRows * 128;          // 16 KB: 128 rows x 64 cols
  static constexpr int kBlkChunk = kBlk * 128;           // rows x 64 cols
  static constexpr int kRowTile = kChunks * kRowChunk;
  static constexpr int kBlkTile = kChunks * kBlkChunk;
  static constexpr int kVecBytes = 1024;                 // L2 and D of up to 128 queries
  // stage: C1 (bf16, then fp16 in the wide layout) | C2 (bf16) | [narrow: C1 as fp16] | vectors
  static constexpr int kStageTiles = kWide ? 2 : 3;
  static constexpr int kStageBytes = kStageTiles * kBlkTile + kVecBytes;
  static_assert(kStageBytes % 1024 == 0, "swizzled tiles need 1 KB alignment");
  // row tiles (R1, R2) of an item; the wide layout double-buffers them so
  // the next item's rows load while this item's last blocks run
  static constexpr int kRBufs = kWide ? (kDefer ? 3 : 2) : 1;
  static constexpr int kR1Off = 0;
  static constexpr int kR2Off = kRowTile;
  static constexpr int kR3Off = 2 * kRowTile;               // O rows (kOwnD)
  static constexpr int kRBufBytes = kRTiles * kRowTile;
  static constexpr int kStageOff = kRBufs * kRBufBytes;
  static constexpr int kBarOff = kStageOff + kStages * kStageBytes;
  static constexpr int kDsumOff = kBarOff + 512;         // 2 items x 2 warpgroups x 128
  static constexpr int kDpartOff = kDsumOff + 2048;      // the same, for D's estimate (kOwnD)
  static constexpr int kSmemBytes = kDpartOff + 2048 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per block");
  // TMEM columns
  static constexpr int kTS = 0;
  static constexpr int kTdP = 128;
  static constexpr int kTAcc1 = 256;                     // dV, or B (dQ kernel)
  static constexpr int kTAcc2 = 256 + DP;                // dK or dQ
  static constexpr int kTP = 384;                        // wide layout only
  static constexpr int kTdS = 448;                       // wide layout only
  static_assert(kWide || DP == 128, "head dims pad to 64 or 128");
};

struct BwdBars {
  uint64_t r_full[3], r_empty[3];
  uint64_t c_full[kStagesMax], c_empty[kStagesMax];
  uint64_t vec_full[kStagesMax], conv_full[kStagesMax];
  uint64_t sp_full, sp_free, pd_full, acc_done;   // wide layout
  uint64_t s_full[2], p_full[2];                  // narrow layout
  uint64_t acc_full, acc_free, dsum, dpart;
  uint64_t epi_staged;   // wide layout, bf16 gradients: the staging tiles are written
  uint64_t drain, probe;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(BwdBars) <= 512, "barrier block");

__device__ __forceinline__ void raise_abort(BwdBars* bars, int* status) {
  record_error(status, FA_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&bars->abort) = 1;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* ab,
                                          long long budget) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab, budget));
}

// Static schedule: the li-th item of this CTA (see the header); -1 when done.
__device__ __forceinline__ int item_index(int li, int num_items) {
  const long long G = gridDim.x, c = blockIdx.x;
  const long long base = static_cast<long long>(li) * G;
  if (base >= num_items) return -1;
  const bool reverse = (li & 1) && base + G <= num_items;
  const long long it = base + (reverse ? G - 1 - c : c);
  return it < num_items ? static_cast<int>(it) : -1;
}

struct Item {
  int b, h, row0, i0, nb;   // streamed blocks [i0, i0 + nb)
};

template <bool kDkDv, bool kCausal, int kBlk>
__device__ __forceinline__ Item decode_item(int it, int N, int H) {
  const int ntiles = (N + kRows - 1) / kRows;
  const int nblocks = (N + kBlk - 1) / kBlk;
  const int bh = it / ntiles, traw = it % ntiles;
  // within a head the longest tile first: dK/dV tiles near the start see the
  // most queries (causal), dQ tiles near the end see the most keys
  const int tile = kDkDv ? traw : (ntiles - 1 - traw);
  Item w;
  w.b = bh / H;
  w.h = bh % H;
  w.row0 = tile * kRows;
  int i1;
  if (kDkDv) {
    w.i0 = kCausal ? (w.row0 / kBlk) : 0;
    i1 = nblocks;
  } else {
    w.i0 = 0;
    i1 = kCausal ? min(nblocks, (w.row0 + kRows + kBlk - 1) / kBlk) : nblocks;
  }
  w.nb = i1 - w.i0;
  return w;
}

// Store 32-column groups [col0, col0 + ncols) of this thread's accumulator row
// at TMEM address `acc`, as mult * (acc + corr * acc_b) (acc_b read only when
// kCorr), to a row of d elements of type float or bf16.
template <bool kF32, bool kCorr, bool kF16>
__device__ __forceinline__ void store_acc_cols(uint32_t acc, uint32_t acc_b, float corr, int col0,
                                               int ncols, float mult, void* row_ptr, int d,
                                               bool store) {
  for (int cc = col0; cc < col0 + ncols; cc += 32) {
    uint32_t r[32];
    __syncwarp();   // the stores below are per-thread; tcgen05.ld is collective
    tmem_ld32(acc + cc, r);
    tmem_ld_wait(r);
    if (kCorr) {
      uint32_t rb[32];
      tmem_ld32(acc_b + cc, rb);
      tmem_ld_wait(rb);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        r[i] = __float_as_uint(fmaf(corr, __uint_as_float(rb[i]), __uint_as_float(r[i])));
    }
    if (!store) continue;
    if (kF32) {
      uint4* out = static_cast<uint4*>(row_ptr);
#pragma unroll
      for (int qv = 0; qv < 8; ++qv) {
        const int col = cc + qv * 4;
        if (col < d) {
          uint4 v;
          v.x = __float_as_uint(__uint_as_float(r[qv * 4 + 0]) * mult);
          v.y = __float_as_uint(__uint_as_float(r[qv * 4 + 1]) * mult);
          v.z = __float_as_uint(__uint_as_float(r[qv * 4 + 2]) * mult);
          v.w = __float_as_uint(__uint_as_float(r[qv * 4 + 3]) * mult);
          out[col / 4] = v;
        }
      }
    } else {
      uint4* out = static_cast<uint4*>(row_ptr);
#pragma unroll
      for (int qv = 0; qv < 4; ++qv) {
        const int col = cc + qv * 8;
        if (col < d) {
          uint4 v;
          v.x = pack16x2<kF16>(__uint_as_float(r[qv * 8 + 0]) * mult,
                            __uint_as_float(r[qv * 8 + 1]) * mult);
          v.y = pack16x2<kF16>(__uint_as_float(r[qv * 8 + 2]) * mult,
                            __uint_as_float(r[qv * 8 + 3]) * mult);
          v.z = pack16x2<kF16>(__uint_as_float(r[qv * 8 + 4]) * mult,
                            __uint_as_float(r[qv * 8 + 5]) * mult);
          v.w = pack16x2<kF16>(__uint_as_float(r[qv * 8 + 6]) * mult,
                            __uint_as_float(r[qv * 8 + 7]) * mult);
          out[col / 8] = v;
        }
      }
    }
  }
}

// Same as store_acc_cols for bf16 output, but into a shared-memory staging
// tile in the TMA box layout (rows of 128 bytes; 16-byte chunk c of row r at
// chunk c ^ (r & 7)); the TMA store clips rows >= N and columns >= d.
template <bool kCorr, bool kF16>
__device__ __forceinline__ void stage_acc_cols(uint32_t acc, uint32_t acc_b, float corr, int col0,
                                               int ncols, float mult, uint8_t* stage, int row) {
  for (int cc = col0; cc < col0 + ncols; cc += 32) {
    uint32_t r[32];
    __syncwarp();   // tcgen05.ld is warp-collective
    tmem_ld32(acc + cc, r);
    tmem_ld_wait(r);
    if (kCorr) {
      uint32_t rb[32];
      tmem_ld32(acc_b + cc, rb);
      tmem_ld_wait(rb);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        r[i] = __float_as_uint(fmaf(corr, __uint_as_float(rb[i]), __uint_as_float(r[i])));
    }
#pragma unroll
    for (int qv = 0; qv < 4; ++qv) {
      const int chunk = (cc >> 3) + qv;   // 16-byte chunk (8 columns) of the row
      uint4 v;
      v.x = pack16x2<kF16>(__uint_as_float(r[qv * 8 + 0]) * mult, __uint_as_float(r[qv * 8 + 1]) * mult);
      v.y = pack16x2<kF16>(__uint_as_float(r[qv * 8 + 2]) * mult, __uint_as_float(r[qv * 8 + 3]) * mult);
      v.z = pack16x2<kF16>(__uint_as_float(r[qv * 8 + 4]) * mult, __uint_as_float(r[qv * 8 + 5]) * mult);
      v.w = pack16x2<kF16>(__uint_as_float(r[qv * 8 + 6]) * mult, __uint_as_float(r[qv * 8 + 7]) * mult);
      *reinterpret_cast<uint4*>(stage + row * 128 + ((chunk ^ (row & 7)) << 4)) = v;
    }
  }
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
  const float lo = __uint_as_float(x << 16);
  const float hi = __uint_as_float(x & 0xffff0000u);
  return pack_f16x2(lo, hi);
}

template <int DP, bool kCausal, bool kDkDv, bool kF32Grad, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmR1, const __grid_constant__ CUtensorMap tmR2,
                  const __grid_constant__ CUtensorMap tmC1, const __grid_constant__ CUtensorMap tmC2,
                  const __grid_constant__ CUtensorMap tmG1, const __grid_constant__ CUtensorMap tmG2,
                  const __grid_constant__ CUtensorMap tmR3, const BwdParams p) {
  using Cfg = BwdCfg<DP, kDkDv>;
  // S/dP, acc1 and acc2 from three issuing warps (1, 3, 2): the wide dQ
  // kernels and the causal wide dK/dV kernel (the fp16 copies are made by the
  // element-wise warps; in that dK/dV kernel warp 2 also writes the
  // per-query vectors).  The non-causal dK/dV kernel measured faster with
  // two (warp 1: S/dP and acc1) and warp 3 writing the vectors.
  constexpr bool kThree = Cfg::kWide && (!kDkDv || kCausal);
  constexpr int S = Cfg::kStages;
  constexpr int kBlk = Cfg::kBlk;
  constexpr bool kWide = Cfg::kWide;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + Cfg::kBarOff);
  float* dsum = reinterpret_cast<float*>(smem + Cfg::kDsumOff);
  float* dpart = reinterpret_cast<float*>(smem + Cfg::kDpartOff);
  const volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int N = p.N, H = p.H;
  const int num_items = ((N + kRows - 1) / kRows) * p.B * H;

  // ---- setup ----
  if (threadIdx.x == 0) {
    for (int b = 0; b < 3; ++b) {
      mbar_init(&bars->r_full[b], 1);
      mbar_init(&bars->r_empty[b], 1);
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars->c_full[s], 1);
      mbar_init(&bars->c_empty[s], kWide ? 2 : 1);   // one commit per MMA warp
      mbar_init(&bars->vec_full[s], 32);
      // who makes the fp16 copy: wide layout: the 256 element-wise threads;
      // narrow: warp 3
      mbar_init(&bars->conv_full[s], kWide ? 256 : 32);
    }
    mbar_init(&bars->sp_full, 1);
    mbar_init(&bars->sp_free, 256);
    mbar_init(&bars->pd_full, 256);
    mbar_init(&bars->acc_done, 2);   // wide layout: one commit per MMA warp
    for (int g = 0; g < 2; ++g) {
      mbar_init(&bars->s_full[g], 1);
      mbar_init(&bars->p_full[g], 128);
    }
    mbar_init(&bars->acc_full, kWide ? 2 : 1);
    mbar_init(&bars->acc_free, 256);
    mbar_init(&bars->dsum, 256);
    mbar_init(&bars->dpart, 256);
    mbar_init(&bars->epi_staged, 256);
    mbar_init(&bars->drain, kThree ? 3 : (kWide ? 2 : 1));   // one commit per MMA warp
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
    if (threadIdx.x == 0 && !mbar_wait(&bars->probe, 0, abort_flag, kProbeBudget))
      raise_abort(bars, p.status);
    __syncthreads();
    run = false;
  }

  uint8_t* sR1 = smem + Cfg::kR1Off;
  uint8_t* sR2 = smem + Cfg::kR2Off;
  auto stage_c1 = [&](int s) { return smem + Cfg::kStageOff + s * Cfg::kStageBytes; };
  auto stage_c2 = [&](int s) { return stage_c1(s) + Cfg::kBlkTile; };
  auto stage_c1h = [&](int s) { return Cfg::kWide ? stage_c1(s) : stage_c1(s) + 2 * Cfg::kBlkTile; };
  auto stage_vec = [&](int s) {
    return reinterpret_cast<float*>(stage_c1(s) + Cfg::kStageTiles * Cfg::kBlkTile);
  };

  // fp16 copy of part [v0, v1) (16-byte units) of stage s's C1 tile (in place in the
  // wide layout, once the block's S has been computed), same
  // swizzled layout; the lanes of one warp share the range
  // (threads: tid = 0 .. nthr-1 share the range)
  auto convert_c1 = [&](int s, int v0, int v1, int tid, int nthr) {
    const uint4* src = reinterpret_cast<const uint4*>(stage_c1(s));
    uint4* dst = reinterpret_cast<uint4*>(stage_c1h(s));
#pragma unroll 4
    for (int i = v0 + tid; i < v1; i += nthr) {
      uint4 v = src[i];
      v.x = bf16x2_to_f16x2(v.x);
      v.y = bf16x2_to_f16x2(v.y);
      v.z = bf16x2_to_f16x2(v.z);
      v.w = bf16x2_to_f16x2(v.w);
      dst[i] = v;
    }
    fence_proxy_async_smem();   // make the copy visible to the tensor cores
  };
  constexpr int kVecs = Cfg::kBlkTile / 16;   // 16-byte units of a C1 tile

  // dK/dV kernel: the per-query -L2 and -D of each streamed block, written
  // to the stage by one warp (narrow layout: warp 2; wide causal: warp 2, the
  // acc2 issuer, one block ahead of its accumulations; wide non-causal: warp 3).  A cursor walks this
  // CTA's blocks; each step reads its block's L and D (two independent
  // loads, in flight while the warp waits for the stage) and writes them.  A
  // block's vectors sit in their own part of the stage (which TMA does not
  // write) and go in as soon as the stage's previous round has been released.
  constexpr int kU = kBlk / 32;
  int v_it = -1, v_li = 0, v_t = 0, v_c = 0;
  Item v_w{};
  auto vec_begin = [&]() {
    v_it = item_index(0, num_items);
    if (v_it >= 0) v_w = decode_item<kDkDv, kCausal, kBlk>(v_it, N, H);
  };
  // write the cursor's block and advance; false if a wait gave up
  auto vec_step = [&]() -> bool {
    if (v_it < 0) return true;
    float L[kU], Dv[kU];
    const size_t hb = (static_cast<size_t>(v_w.b) * H + v_w.h) * N;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int q = (v_w.i0 + v_t) * kBlk + u * 32 + lane;
      L[u] = -INFINITY;   // padded query: P = 0
      Dv[u] = 0.0f;
      if (q < N) {
        L[u] = p.lse[hb + q];
        Dv[u] = p.D[hb + q];
      }
    }
    const int s = v_c % S, round = v_c / S;
    if (round > 0 &&
        !warp_wait(&bars->c_empty[s], (round - 1) & 1, abort_flag, kWaitBudget))
      return false;
    float* vec = stage_vec(s);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      // a fully masked query (L = -inf) gets P = 0 and dS = 0
      const bool live = L[u] != -INFINITY;
      vec[u * 32 + lane] = live ? -L[u] * kLog2e : -INFINITY;   // -L2: exponent s c + (-L2)
      vec[kBlk + u * 32 + lane] = live ? -Dv[u] : 0.0f;         // -D
    }
    mbar_arrive(&bars->vec_full[s]);
    ++v_c;
    if (++v_t >= v_w.nb) {
      v_t = 0;
      v_it = item_index(++v_li, num_items);
      if (v_it >= 0) v_w = decode_item<kDkDv, kCausal, kBlk>(v_it, N, H);
    }
    return true;
  };

  // Role bodies; each runs inside the branch that sets its register budget
  // (setmaxnreg: the element-wise warps hold S, dP, P and dS of a row).
  auto helper_roles = [&]() {
  if (run && warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tmR1);
      tma_prefetch_desc(&tmR2);
      tma_prefetch_desc(&tmC1);
      tma_prefetch_desc(&tmC2);
      int c = 0, li = 0;
      bool ok = true;
      for (int it = item_index(0, num_items); it >= 0 && ok; it = item_index(li, num_items)) {
        const Item w = decode_item<kDkDv, kCausal, kBlk>(it, N, H);
        // row buffer rb, its use number ru
        const int rb = li % Cfg::kRBufs, ru = li / Cfg::kRBufs;
        if (ru > 0 &&
            !mbar_wait(&bars->r_empty[rb], (ru - 1) & 1, abort_flag, kWaitBudget)) {
          ok = false;
          break;
        }
        uint8_t* r1 = sR1 + rb * Cfg::kRBufBytes;
        uint8_t* r2 = sR2 + rb * Cfg::kRBufBytes;
        mbar_arrive_expect_tx(&bars->r_full[rb], Cfg::kRTiles * Cfg::kRowTile);
        for (int ch = 0; ch < Cfg::kChunks; ++ch) {
          tma_load_4d(r1 + ch * Cfg::kRowChunk, &tmR1, &bars->r_full[rb], ch * 64, w.h, w.row0,
                      w.b);
          tma_load_4d(r2 + ch * Cfg::kRowChunk, &tmR2, &bars->r_full[rb], ch * 64, w.h, w.row0,
                      w.b);
          if constexpr (Cfg::kOwnD)
            tma_load_4d(sR1 + rb * Cfg::kRBufBytes + Cfg::kR3Off + ch * Cfg::kRowChunk, &tmR3,
                        &bars->r_full[rb], ch * 64, w.h, w.row0, w.b);
        }
        ++li;
        for (int t = 0; t < w.nb; ++t) {
          const int s = c % S, round = c / S;
          if (round > 0 &&
              !mbar_wait(&bars->c_empty[s], (round - 1) & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
          const int r = (w.i0 + t) * kBlk;
          mbar_arrive_expect_tx(&bars->c_full[s], 2 * Cfg::kBlkTile);
          for (int ch = 0; ch < Cfg::kChunks; ++ch) {
            tma_load_4d(stage_c1(s) + ch * Cfg::kBlkChunk, &tmC1, &bars->c_full[s], ch * 64, w.h,
                        r, w.b);
            tma_load_4d(stage_c2(s) + ch * Cfg::kBlkChunk, &tmC2, &bars->c_full[s], ch * 64, w.h,
                        r, w.b);
          }
          ++c;
        }
      }
      if (!ok) raise_abort(bars, p.status);
      for (int x = max(0, c - S); x < c; ++x)
        mbar_wait(&bars->c_full[x % S], (x / S) & 1, nullptr, kDrainBudget);
      for (int x = max(0, li - Cfg::kRBufs); x < li; ++x)
        mbar_wait(&bars->r_full[x % Cfg::kRBufs], (x / Cfg::kRBufs) & 1, nullptr, kDrainBudget);
    }
    __syncwarp();
  } else if (run && (warp == 1 || (kWide && warp == 2) || (kThree && warp == 3))) {
    // ============ MMA issuers (whole warp waits, lane 0 issues) ============
    const uint32_t leader = (lane == 0) ? 1u : 0u;
    constexpr uint32_t kIdescSP = idesc16<kF16>(kRows, kBlk, false, false);
    constexpr uint32_t kIdescAccBf = idesc16<kF16>(kRows, DP, false, true);   // dV += P dO
    constexpr uint32_t kIdescAccH = idesc_f16(kRows, DP, false, true);
    const int nks = (p.d + 15) / 16;
    // descriptor bases; offsets advance the 16-byte start-address field
    const uint64_t dR1 = sdesc_sw128(smem_u32(sR1), 16, 1024);
    const uint64_t dR2 = sdesc_sw128(smem_u32(sR2), 16, 1024);
    const uint64_t dC1 = sdesc_sw128(smem_u32(stage_c1(0)), 16, 1024);
    const uint64_t dC2 = sdesc_sw128(smem_u32(stage_c2(0)), 16, 1024);
    // fp16 view of the streamed C1 tile: the copy, or (fp16 storage) the tile itself
    const uint64_t dC1hMN = sdesc_sw128(smem_u32(kF16 ? stage_c1(0) : stage_c1h(0)),
                                        Cfg::kBlkChunk, 1024);
    const uint64_t dC2MN = sdesc_sw128(smem_u32(stage_c2(0)), Cfg::kBlkChunk, 1024);

    // S and dP of global block cb into TMEM column offset `col`, rows from
    // row buffer rb
    auto issue_sp = [&](int cb, int col, int rb) {
      const uint64_t so = static_cast<uint64_t>(((cb % S) * Cfg::kStageBytes) >> 4);
      const uint64_t rbo = static_cast<uint64_t>((rb * Cfg::kRBufBytes) >> 4);
      auto step = [&](int kk) {
        const uint64_t ro = static_cast<uint64_t>(((kk >> 2) * Cfg::kRowChunk + (kk & 3) * 32) >> 4);
        const uint64_t co = static_cast<uint64_t>(((kk >> 2) * Cfg::kBlkChunk + (kk & 3) * 32) >> 4);
        mma_ss(tmem + Cfg::kTS + col, dR1 + rbo + ro, dC1 + so + co, kIdescSP, kk > 0);
        mma_ss(tmem + Cfg::kTdP + col, dR2 + rbo + ro, dC2 + so + co, kIdescSP, kk > 0);
      };
      if (leader) {
        // d = DP in the three-issuer kernels: fully unrolled with constant
        // offsets (short issue stream); elsewhere the loop, with descriptors
        // advanced in place
        if (kThree && nks == DP / 16) {
#pragma unroll
          for (int kk = 0; kk < DP / 16; ++kk) step(kk);
        } else {
          // descriptors advanced in place: +32 B per K=16 step inside a
          // 64-column chunk, then on to the next chunk
          uint64_t a1 = dR1 + rbo, a2 = dR2 + rbo, b1 = dC1 + so, b2 = dC2 + so;
          constexpr uint64_t kRowJump = (Cfg::kRowChunk - 96) >> 4;
          constexpr uint64_t kBlkJump = (Cfg::kBlkChunk - 96) >> 4;
          for (int kk = 0; kk < nks; ++kk) {
            mma_ss(tmem + Cfg::kTS + col, a1, b1, kIdescSP, kk > 0);
            mma_ss(tmem + Cfg::kTdP + col, a2, b2, kIdescSP, kk > 0);
            const bool wrap = (kk & 3) == 3;
            a1 += wrap ? kRowJump : 2;
            a2 += wrap ? kRowJump : 2;
            b1 += wrap ? kBlkJump : 2;
            b2 += wrap ? kBlkJump : 2;
          }
        }
      }
      __syncwarp();
    };
    // accumulating MMAs of global block cb; P and dS at TMEM columns pcol,
    // dcol.  parts: 1 = acc1 only, 2 = acc2 only, 3 = both (interleaved).
    //   acc1: dV += P dO_i (bf16)  or  B += P K_j (fp16)
    //   acc2: dK += dS Q_i         or  dQ += dS K_j   (fp16)
    auto issue_acc = [&](int cb, bool first, uint32_t pcol, uint32_t dcol, int parts) {
      const uint64_t so = static_cast<uint64_t>(((cb % S) * Cfg::kStageBytes) >> 4);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk) {
          const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
          const uint32_t pa = tmem + pcol + kk * 8;
          const uint32_t da = tmem + dcol + kk * 8;
          const uint64_t ko = static_cast<uint64_t>((kk * 2048) >> 4);
          if (parts & 1) {
            if (kDkDv)
              mma_ts(tmem + Cfg::kTAcc1, pa, dC2MN + so + ko, kIdescAccBf, acc);
            else
              mma_ts(tmem + Cfg::kTAcc1, pa, dC1hMN + so + ko, kIdescAccH, acc);
          }
          if (parts & 2) mma_ts(tmem + Cfg::kTAcc2, da, dC1hMN + so + ko, kIdescAccH, acc);
        }
        mma_commit(&bars->c_empty[cb % S]);
      }
      __syncwarp();
    };
    auto wait_c = [&](int cb) {
      return warp_wait(&bars->c_full[cb % S], (cb / S) & 1, abort_flag, kWaitBudget);
    };
    // need_conv: the MMAs read the fp16 copy of the streamed C1 tile
    auto wait_acc_inputs = [&](int cb, bool item_first, int li, bool need_conv = true) {
      bool ok = !need_conv || kF16 ||
                warp_wait(&bars->conv_full[cb % S], (cb / S) & 1, abort_flag, kWaitBudget);
      // the first accumulation of an item overwrites the accumulators: the
      // previous item's epilogue must have read them
      if (ok && item_first && li > 0)
        ok = warp_wait(&bars->acc_free, (li - 1) & 1, abort_flag, kWaitBudget);
      return ok;
    };

    int c = 0, li = 0;
    int nsp = 0;   // wide: S/dP groups issued; narrow: unused
    int npd = 0;   // wide: pd_full phases consumed
    bool ok = true;
    for (int it = item_index(0, num_items); it >= 0 && ok; it = item_index(++li, num_items)) {
      const Item w = decode_item<kDkDv, kCausal, kBlk>(it, N, H);
      if (kThree && warp == 3) {
        // third MMA warp (causal dQ kernel): the acc1 accumulations of every
        // block.  S/dP (warp 1), acc1 (warp 3) and acc2 (warp 2) come from
        // three threads, so no chain of MMAs waits behind another in program
        // order.
        for (int t = 0; t < w.nb; ++t) {
          const int cb = c + t;
          if (!warp_wait(&bars->pd_full, npd & 1, abort_flag, kWaitBudget) ||
              !wait_acc_inputs(cb, t == 0, li, !kDkDv)) {
            ok = false;
            break;
          }
          ++npd;
          tc_fence_after();
          issue_acc(cb, t == 0, Cfg::kTP, Cfg::kTdS, 1);
          mma_commit_w(&bars->acc_done, leader);
          if (t == w.nb - 1) mma_commit_w(&bars->acc_full, leader);
        }
        c += w.nb;
        continue;
      }
      if (kWide && warp == 2) {
        // second MMA warp (wide layout): the acc2 accumulations of every
        // block, concurrently with the acc1 ones (warp 3 with kThree, else
        // warp 1; a single issuing thread cannot keep the tensor pipe busy
        // with N = 64 MMAs).  In the dK/dV kernel it first writes the next
        // block's per-query vectors (the first block's before the loop).
        if (kDkDv && kThree && li == 0) {
          vec_begin();
          if (!vec_step()) {
            ok = false;
            break;
          }
        }
        for (int t = 0; t < w.nb; ++t) {
          const int cb = c + t;
          if (kDkDv && kThree && !vec_step()) {
            ok = false;
            break;
          }
          if (!warp_wait(&bars->pd_full, npd & 1, abort_flag, kWaitBudget) ||
              !wait_acc_inputs(cb, t == 0, li)) {
            ok = false;
            break;
          }
          ++npd;
          tc_fence_after();
          issue_acc(cb, t == 0, Cfg::kTP, Cfg::kTdS, 2);
          mma_commit_w(&bars->acc_done, leader);
          if (t == w.nb - 1) mma_commit_w(&bars->acc_full, leader);
        }
        c += w.nb;
        continue;
      }
      const int rb = li % Cfg::kRBufs;
      if (!warp_wait(&bars->r_full[rb], (li / Cfg::kRBufs) & 1, abort_flag, kWaitBudget)) {
        ok = false;
        break;
      }
      if constexpr (kWide) {
        auto next_sp = [&](int cb) -> bool {
          if (!wait_c(cb)) return false;
          if (nsp > 0 && !warp_wait(&bars->sp_free, (nsp - 1) & 1, abort_flag, kWaitBudget))
            return false;
          tc_fence_after();
          issue_sp(cb, 0, rb);
          mma_commit_w(&bars->sp_full, leader);
          ++nsp;
          return true;
        };
        if constexpr (kThree) {
          // S/dP only, each block's as soon as the element-wise warps hold
          // the previous one in registers (warp 3 issues acc1)
          for (int t = 0; t < w.nb && ok; ++t)
            if (!next_sp(c + t)) ok = false;
          if (!ok) break;
        } else {
          // S/dP of the next block, then acc1 of this one
          if (!next_sp(c)) { ok = false; break; }
          for (int t = 0; t < w.nb; ++t) {
            const int cb = c + t;
            if (t + 1 < w.nb && !next_sp(cb + 1)) { ok = false; break; }
            if (!warp_wait(&bars->pd_full, npd & 1, abort_flag, kWaitBudget) ||
                !wait_acc_inputs(cb, t == 0, li, !kDkDv)) {
              ok = false;
              break;
            }
            ++npd;
            tc_fence_after();
            issue_acc(cb, t == 0, Cfg::kTP, Cfg::kTdS, 1);
            mma_commit_w(&bars->acc_done, leader);
            if (t == w.nb - 1) mma_commit_w(&bars->acc_full, leader);
          }
        }
      } else {
        // narrow: S/dP of global block cb go to buffer cb & 1; warpgroup cb & 1
        // forms P and dS in place
        for (int t = 0; t <= w.nb && ok; ++t) {
          const int cb = c + t;
          if (t < w.nb) {
            if (!wait_c(cb)) { ok = false; break; }
            tc_fence_after();
            issue_sp(cb, (cb & 1) * kBlk, rb);
            mma_commit_w(&bars->s_full[cb & 1], leader);
            if (t == w.nb - 1) mma_commit_w(&bars->r_empty[rb], leader);
          }
          if (t >= 1) {
            const int pb = cb - 1;
            if (!warp_wait(&bars->p_full[pb & 1], (pb >> 1) & 1, abort_flag, kWaitBudget) ||
                !wait_acc_inputs(pb, t == 1, li)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_acc(pb, t == 1, Cfg::kTS + (pb & 1) * kBlk, Cfg::kTdP + (pb & 1) * kBlk, 3);
            if (t == w.nb) mma_commit_w(&bars->acc_full, leader);
          }
        }
      }
      c += w.nb;
    }
    if (!ok && leader) raise_abort(bars, p.status);
    mma_commit_w(&bars->drain, leader);
    mbar_wait(&bars->drain, 0, nullptr, kDrainBudget);
    __syncwarp();
  } else if (run && warp == 2) {
    // ===== narrow layout: per-query L and D of each streamed block (dK/dV) =====
    if (kDkDv) {
      bool ok = true;
      vec_begin();
      while (ok && v_it >= 0) ok = vec_step();
      if (!ok && lane == 0) raise_abort(bars, p.status);
    }
    __syncwarp();
  } else if (run && warp == 3) {
    // ============ narrow layout: fp16 copy of each streamed C1 tile ============
    // (same swizzled layout).  Wide layout: the element-wise warps make the
    // copy, and this warp is the third MMA issuer, or (non-causal dK/dV
    // kernel) writes the per-query vectors.
    int c = 0, li = 0;
    bool ok = true;
    if constexpr (kWide && kDkDv) {
      vec_begin();
      while (ok && v_it >= 0) ok = vec_step();
    } else if constexpr (!kWide) {
      for (int it = item_index(0, num_items); it >= 0 && ok; it = item_index(++li, num_items)) {
        const Item w = decode_item<kDkDv, kCausal, kBlk>(it, N, H);
        for (int t = 0; t < w.nb; ++t, ++c) {
          const int s = c % S;
          if (!warp_wait(&bars->c_full[s], (c / S) & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
          if (kF16) continue;   // fp16 storage: the tile itself is the operand
          convert_c1(s, kWide ? kVecs / 2 : 0, kVecs, lane, 32);
          mbar_arrive(&bars->conv_full[s]);
        }
      }
    }
    if (!ok && lane == 0) raise_abort(bars, p.status);
    __syncwarp();
  }
  };
  auto elementwise_role = [&]() {
  if (run) {
    // ======================= element-wise warpgroups =======================
    const int g = (warp - 4) / 4;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = p.scale_log2;
    // wide: this warpgroup's 64 columns of every block; narrow: buffer g
    const uint32_t tS = tmem + lane_base + Cfg::kTS + g * 64;
    const uint32_t tdP = tmem + lane_base + Cfg::kTdP + g * 64;
    const uint32_t tP = tmem + lane_base + (kWide ? Cfg::kTP + g * 32 : Cfg::kTS + g * 64);
    const uint32_t tdS = tmem + lane_base + (kWide ? Cfg::kTdS + g * 32 : Cfg::kTdP + g * 64);
    const int colg = kWide ? g * 64 : 0;    // first block column this warpgroup handles
    int cbase = 0, li = 0;
    int nsp = 0;    // wide: sp_full phases consumed
    // thread 128 (wide layout, bf16 gradients): the row buffer whose staged
    // gradient rows are being stored; it goes back to the producer once the
    // TMA stores have read it, checked a block later so nobody waits for it
    int pend_rb = -1;
    auto release_rows = [&]() {
      if (pend_rb >= 0) {
        bulk_wait_read_all();
        mbar_arrive(&bars->r_empty[pend_rb]);
        pend_rb = -1;
      }
    };
    bool ok = true;
    // dQ kernel: this thread's query L and D of an item, read one item ahead
    // (two independent loads) so the first block's exponent does not wait
    auto load_row = [&](int it2, float& L, float& Dv) {
      L = -INFINITY;
      Dv = 0.0f;
      if (it2 < 0) return;
      const Item w2 = decode_item<kDkDv, kCausal, kBlk>(it2, N, H);
      const int g2 = w2.row0 + row;
      if (g2 < N) {
        const size_t hb2 = (static_cast<size_t>(w2.b) * H + w2.h) * N;
        L = p.lse[hb2 + g2];
        if (!Cfg::kOwnD) Dv = p.D[hb2 + g2];
      }
    };
    // An item's epilogue: wait for its last accumulations, then this
    // warpgroup stores half of the accumulator columns (dQ: with the
    // correction corr of its D refinement).  The wide dK/dV kernel defers it
    // to the next item's first block, after that block's element-wise math
    // and before its P and dS overwrite the TMEM the accumulations read.
    auto epilogue = [&](const Item& ew, int eli, float corr) -> bool {
      if (!warp_wait(&bars->acc_full, eli & 1, abort_flag, kWaitBudget)) return false;
      tc_fence_after();
      const int egrow = ew.row0 + row;
      const bool store = egrow < N;
      const size_t roff = ((static_cast<size_t>(ew.b) * N + (store ? egrow : 0)) * H + ew.h) *
                          static_cast<size_t>(p.d);
      const int half_cols = DP / 2;
      const int cbeg = g * half_cols;
      auto row_ptr = [&](void* base) -> void* {
        return kF32Grad ? static_cast<void*>(static_cast<float*>(base) + roff)
                        : static_cast<void*>(static_cast<__nv_bfloat16*>(base) + roff);
      };
      if constexpr (kWide && !kF32Grad) {
        // Wide layout, bf16 gradients: stage the rows in this item's row
        // buffer (its last S/dP MMAs have completed, acc_full says so) and
        // write them with TMA tensor stores; the buffer is released to the
        // producer once the stores have read it.
        const int rb = eli % Cfg::kRBufs;
        uint8_t* st1 = sR1 + rb * Cfg::kRBufBytes;
        uint8_t* st2 = sR2 + rb * Cfg::kRBufBytes;
        if (kDkDv) {
          stage_acc_cols<false, kF16>(tmem + lane_base + Cfg::kTAcc1, 0, 0.0f, cbeg, half_cols, 1.0f,
                                st1, row);
          stage_acc_cols<false, kF16>(tmem + lane_base + Cfg::kTAcc2, 0, 0.0f, cbeg, half_cols, p.scale,
                                st2, row);
        } else {
          stage_acc_cols<true, kF16>(tmem + lane_base + Cfg::kTAcc2, tmem + lane_base + Cfg::kTAcc1, corr,
                               cbeg, half_cols, p.scale, st1, row);
        }
        fence_proxy_async_smem();   // the TMA engine reads what the threads wrote
        tc_fence_before();
        mbar_arrive(&bars->acc_free);
        mbar_arrive(&bars->epi_staged);
        bool sok = true;
        if (threadIdx.x == 128) {
          if (!mbar_wait(&bars->epi_staged, eli & 1, abort_flag, kWaitBudget)) {
            sok = false;
          } else {
            tma_store_4d(&tmG1, st1, 0, ew.h, ew.row0, ew.b);
            if (kDkDv) tma_store_4d(&tmG2, st2, 0, ew.h, ew.row0, ew.b);
            bulk_commit_group();
            pend_rb = rb;   // released once the stores have read it (next block)
          }
        }
        if (!__all_sync(0xffffffffu, sok)) return false;
      } else {
        if (kDkDv) {
          store_acc_cols<kF32Grad, false, kF16>(tmem + lane_base + Cfg::kTAcc1, 0, 0.0f, cbeg,
                                          half_cols, 1.0f, row_ptr(p.dv), p.d, store);
          store_acc_cols<kF32Grad, false, kF16>(tmem + lane_base + Cfg::kTAcc2, 0, 0.0f, cbeg,
                                          half_cols, p.scale, row_ptr(p.dk), p.d, store);
        } else {
          store_acc_cols<kF32Grad, true, kF16>(tmem + lane_base + Cfg::kTAcc2,
                                         tmem + lane_base + Cfg::kTAcc1, corr, cbeg, half_cols,
                                         p.scale, row_ptr(p.dq), p.d, store);
        }
        tc_fence_before();
        mbar_arrive(&bars->acc_free);
        // wide layout, fp32 gradients: the row buffer is free (acc_full)
        if (kWide && threadIdx.x == 128) mbar_arrive(&bars->r_empty[eli % Cfg::kRBufs]);
      }
      return true;
    };
    // wide dK/dV kernel: the item whose epilogue is still to run
    bool epi_pend = false;
    Item ew_pend{};
    int eli_pend = 0;
    float L_nx = -INFINITY, D_nx = 0.0f;
    if (!kDkDv) load_row(item_index(0, num_items), L_nx, D_nx);
    // wide dQ kernel: D's first estimate, the float32 dot of this query's dO
    // and O rows (bf16 or fp16, in the item's row buffer, 128-byte swizzle);
    // warpgroup g takes 16-byte chunks [4g, 4g + 4) of the row
    auto row_dot = [&](int rb) -> float {
      const uint8_t* rdo = sR2 + rb * Cfg::kRBufBytes + row * 128;
      const uint8_t* ro = sR1 + rb * Cfg::kRBufBytes + Cfg::kR3Off + row * 128;
      uint64_t acc[4] = {0, 0, 0, 0};   // four packed f32x2 chains (+0.0f pairs)
#pragma unroll
      for (int cq = 0; cq < 4; ++cq) {
        const int ck = 4 * g + cq;
        const int off = (ck ^ (row & 7)) << 4;
        const uint4 a = *reinterpret_cast<const uint4*>(rdo + off);
        const uint4 b = *reinterpret_cast<const uint4*>(ro + off);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 x, y;
          if constexpr (kF16) {
            x = __half22float2(*reinterpret_cast<const __half2*>(&av[i]));
            y = __half22float2(*reinterpret_cast<const __half2*>(&bv[i]));
          } else {
            x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[i]));
            y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bv[i]));
          }
          acc[i] = f2_fma(f2_pack(x.x, x.y), f2_pack(y.x, y.y), acc[i]);
        }
      }
      const uint64_t s2 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
      return f2_lo(s2) + f2_hi(s2);
    };
    for (int it = item_index(0, num_items); it >= 0 && ok; it = item_index(++li, num_items)) {
      const Item w = decode_item<kDkDv, kCausal, kBlk>(it, N, H);
      const int grow = w.row0 + row;      // query (dQ) or key (dK/dV)
      const size_t hb = (static_cast<size_t>(w.b) * H + w.h) * N;
      float l2_row = INFINITY, d_row = 0.0f;          // dQ kernel: this query's L, D~
      bool live_row = false;
      if (!kDkDv) {
        const float L = L_nx;
        float Dv = D_nx;
        load_row(item_index(li + 1, num_items), L_nx, D_nx);
        if constexpr (Cfg::kOwnD) {
          // the item's rows have landed (also what the MMA warp waits for)
          const int rb = li % Cfg::kRBufs;
          if (!warp_wait(&bars->r_full[rb], (li / Cfg::kRBufs) & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
          // the two warpgroups' halves of the dot, exchanged through shared
          // memory (each item's slot pair alternates)
          float* dp = dpart + (li & 1) * 256;
          dp[g * kRows + row] = row_dot(rb);
          mbar_arrive(&bars->dpart);
          if (!warp_wait(&bars->dpart, li & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
          Dv = dp[row] + dp[kRows + row];
        }
        if (grow < N && L != -INFINITY) {
          live_row = true;
          l2_row = L * kLog2e;
          d_row = Dv;
        }
      }
      float d_acc = 0.0f;                             // dQ kernel: sum_j P_ij dP_ij
      for (int t = 0; t < w.nb; ++t) {
        const int cb = cbase + t;
        if (!kWide && (cb & 1) != g) continue;
        if (kWide) {
          if (!warp_wait(&bars->sp_full, nsp & 1, abort_flag, kWaitBudget)) { ok = false; break; }
          ++nsp;
        } else {
          if (!warp_wait(&bars->s_full[g], (cb >> 1) & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
        }
        const int s = cb % S;
        if (kDkDv &&
            !warp_wait(&bars->vec_full[s], (cb / S) & 1, abort_flag, kWaitBudget)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if constexpr (kDkDv && kWide) {
          // dK/dV, wide layout: each thread takes 4 rows x 16 columns of the
          // warpgroup's 64 (16x256b TMEM loads), so it needs the per-query
          // -L2 and -D of 16 columns instead of 64.  Rows: lane group h
          // (lanes 16h .. 16h+15 of the warp's quarter), rows t/4 and t/4+8
          // of it; columns 8k + 2(t%4) and +1, k = 0..7.
          uint32_t s4[2][32], d4[2][32];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tmem_ld16x256_x8(tS + (static_cast<uint32_t>(16 * h) << 16), s4[h]);
            tmem_ld16x256_x8(tdP + (static_cast<uint32_t>(16 * h) << 16), d4[h]);
          }
          // while the loads are in flight: this block's fp16 copy of C1 for
          // the dK accumulation (the block has landed: its S was computed)
          if (!kF16) {
            convert_c1(s, 0, kVecs, threadIdx.x - 128, 256);
            mbar_arrive(&bars->conv_full[s]);
          }
          tmem_ld_wait(s4[0]);
          tmem_ld_wait(s4[1]);
          tmem_ld_wait(d4[0]);
          tmem_ld_wait(d4[1]);
          tc_fence_before();
          mbar_arrive(&bars->sp_free);
          const int tq = lane & 3, tr = lane >> 2;
          const int col0 = (w.i0 + t) * kBlk + colg;
          // causal: query col0 + c is masked for key grow_r when c < grow_r - col0
          if (kCausal && col0 < w.row0 + kRows - 1) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int lim = w.row0 + quarter * 32 + 16 * h + tr + 8 * e - col0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
#pragma unroll
                  for (int b = 0; b < 2; ++b) {
                    const int cidx = 8 * k + 2 * tq + b;
                    uint32_t& v = s4[h][4 * k + 2 * e + b];
                    v = (cidx < lim) ? __float_as_uint(-INFINITY) : v;
                  }
                }
              }
            }
          }
          const float* vbase = stage_vec(s) + colg + 2 * tq;
          const uint64_t c2 = f2_pack(c, c);
          uint32_t pk4[2][16], dk4[2][16];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 a = *reinterpret_cast<const float2*>(vbase + 8 * k);
            const float2 bq = *reinterpret_cast<const float2*>(vbase + kBlk + 8 * k);
            const uint64_t nl2 = f2_pack(a.x, a.y);
            const uint64_t nd = f2_pack(bq.x, bq.y);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int ri = 4 * k + 2 * e;
                const uint64_t s2 = f2_pack(__uint_as_float(s4[h][ri]), __uint_as_float(s4[h][ri + 1]));
                const uint64_t dp2 = f2_pack(__uint_as_float(d4[h][ri]), __uint_as_float(d4[h][ri + 1]));
                const uint64_t t2 = f2_fma(s2, c2, nl2);
                const float p0 = fast_exp2(f2_lo(t2));
                const float p1 = fast_exp2(f2_hi(t2));
                const uint64_t ds2 = f2_mul(f2_pack(p0, p1), f2_add(dp2, nd));
                pk4[h][2 * k + e] = pack16x2<kF16>(p0, p1);
                dk4[h][2 * k + e] = pack_f16x2(f2_lo(ds2), f2_hi(ds2));
              }
            }
          }
          if (threadIdx.x == 128) release_rows();
          // the previous item's deferred epilogue: its accumulators must be
          // read before this block's P V and dS Q overwrite them
          if (Cfg::kDefer && t == 0 && epi_pend) {
            epi_pend = false;
            if (!epilogue(ew_pend, eli_pend, 0.0f)) {
              ok = false;
              break;
            }
          }
          // P and dS columns are free once the previous block's accumulating
          // MMAs have completed
          if (nsp >= 2 &&
              !warp_wait(&bars->acc_done, nsp & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
          tc_fence_after();
          __syncwarp();   // tcgen05.st is warp-collective
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tmem_st16x128_x8(tP + (static_cast<uint32_t>(16 * h) << 16), pk4[h]);
            tmem_st16x128_x8(tdS + (static_cast<uint32_t>(16 * h) << 16), dk4[h]);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars->pd_full);
          continue;
        }
        uint32_t sr[64], dr[64];
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld32(tdP, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
        tmem_ld32(tdP + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
        // wide dQ kernel: this block's fp16 copy of K for the accumulations
        // (the block has landed: its S was computed), made while the loads
        // are in flight and off the MMA-issuing warps
        if (kWide && !kDkDv && !kF16) {
          convert_c1(s, 0, kVecs, threadIdx.x - 128, 256);
          mbar_arrive(&bars->conv_full[s]);
        }
        tmem_ld_wait(sr);
        tmem_ld_wait(dr);
        if (kWide) {
          // S and dP are in registers: the next block's MMAs may overwrite them
          tc_fence_before();
          mbar_arrive(&bars->sp_free);
        }
        const int col0 = (w.i0 + t) * kBlk + colg;   // first query (dK/dV) or key (dQ)
        // Masked pairs get s = -inf before the exponent (P = 0, dS = 0): a
        // select against a per-row column limit, in blocks that need it.
        //   dK/dV (row = key, column = query): masked when query < key.
        //   dQ (row = query, column = key): masked when key > query or key >= N.
        // Queries >= N in the dK/dV kernel carry -L2 = -inf, which also gives 0.
        if (kDkDv) {
          if (kCausal && col0 < w.row0 + kRows - 1) {
            const int lim = grow - col0;   // columns cl < lim are masked
            // one 32-bit keep mask per 32 columns, a bit select per score
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int sh = lim - 32 * k;   // keep columns 32k + sh ..
              const uint32_t keep = sh <= 0 ? 0xffffffffu : (sh >= 32 ? 0u : (0xffffffffu << sh));
#pragma unroll
              for (int i = 0; i < 32; ++i)
                sr[32 * k + i] = ((keep >> i) & 1u) ? sr[32 * k + i] : __float_as_uint(-INFINITY);
            }
          }
        } else if ((kCausal && col0 + 63 > w.row0) || (col0 + 64 > N)) {
          const int lim = min(kCausal ? grow - col0 : 64, N - 1 - col0);   // cl > lim masked
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int sh = lim - 32 * k;   // keep columns 32k .. 32k + sh
            const uint32_t keep =
                sh >= 31 ? 0xffffffffu : (sh < 0 ? 0u : (0xffffffffu >> (31 - sh)));
#pragma unroll
            for (int i = 0; i < 32; ++i)
              sr[32 * k + i] = ((keep >> i) & 1u) ? sr[32 * k + i] : __float_as_uint(-INFINITY);
          }
        }
        // Element-wise math on packed pairs (f32x2): t = s c - L2,
        // P = 2^t, dS = P (dP - D); the dQ kernel also sums P dP per row.
        // dK/dV: the per-column -L2 and -D come from shared memory (the same
        // values for every row), read 8 columns at a time with 16-byte loads
        // one chunk ahead of their use, so the load latency overlaps the math.
        const float4* nl2v = kDkDv ? reinterpret_cast<const float4*>(stage_vec(s) + colg) : nullptr;
        const float4* ndv = kDkDv ? reinterpret_cast<const float4*>(stage_vec(s) + kBlk + colg)
                                  : nullptr;
        const uint64_t c2 = f2_pack(c, c);
        const uint64_t nl2_row = f2_pack(-l2_row, -l2_row);
        const uint64_t nd_row = f2_pack(-d_row, -d_row);
        uint64_t dacc2 = 0;   // (+0.0f, +0.0f)
        uint32_t pk[32], dk[32];
        float4 vl[2], vd[2];   // the chunk being used
        if (kDkDv) {
          vl[0] = nl2v[0]; vl[1] = nl2v[1];
          vd[0] = ndv[0]; vd[1] = ndv[1];
        }
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {   // 8 columns (4 pairs) per chunk
          float4 nl[2], nn[2];
          if (kDkDv && ch + 1 < 8) {
            nl[0] = nl2v[2 * ch + 2]; nl[1] = nl2v[2 * ch + 3];
            nn[0] = ndv[2 * ch + 2]; nn[1] = ndv[2 * ch + 3];
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i = ch * 4 + q;   // pair index: columns 2i, 2i+1
            uint64_t nl2, nd;
            if (kDkDv) {
              const float4& a4 = vl[q >> 1];
              const float4& d4 = vd[q >> 1];
              nl2 = (q & 1) ? f2_pack(a4.z, a4.w) : f2_pack(a4.x, a4.y);
              nd = (q & 1) ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y);
            } else {
              nl2 = nl2_row;
              nd = nd_row;
            }
            const uint64_t s2 = f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]));
            const uint64_t dp2 = f2_pack(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1]));
            const uint64_t t2 = f2_fma(s2, c2, nl2);
            const float p0 = fast_exp2(f2_lo(t2));
            const float p1 = fast_exp2(f2_hi(t2));
            const uint64_t p2 = f2_pack(p0, p1);
            if (!kDkDv) dacc2 = f2_fma(p2, dp2, dacc2);
            const uint64_t ds2 = f2_mul(p2, f2_add(dp2, nd));
            pk[i] = kDkDv ? pack16x2<kF16>(p0, p1) : pack_f16x2(p0, p1);
            dk[i] = pack_f16x2(f2_lo(ds2), f2_hi(ds2));
          }
          if (kDkDv && ch + 1 < 8) {
            vl[0] = nl[0]; vl[1] = nl[1];
            vd[0] = nn[0]; vd[1] = nn[1];
          }
        }
        if (!kDkDv) d_acc += f2_lo(dacc2) + f2_hi(dacc2);
        if (kWide) {
          if (threadIdx.x == 128) release_rows();
          // P and dS columns are free once the previous block's accumulating
          // MMAs have completed
          if (nsp >= 2 &&
              !warp_wait(&bars->acc_done, nsp & 1, abort_flag, kWaitBudget)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        __syncwarp();   // tcgen05.st is warp-collective
        tmem_st32(tP, pk);
        tmem_st32(tdS, dk);
        tmem_st_wait();
        tc_fence_before();
        if (kWide) mbar_arrive(&bars->pd_full);
        else mbar_arrive(&bars->p_full[g]);
      }
      if (!ok) break;

      // ---- epilogue: this warpgroup stores half of the accumulator columns ----
      float corr = 0.0f;
      if (!kDkDv) {
        // Combine the two warpgroups' partial sums of D_i = sum_j P_ij dP_ij.
        float* ds_item = dsum + (li & 1) * 256;
        ds_item[g * kRows + row] = d_acc;
        mbar_arrive(&bars->dsum);
        if (!warp_wait(&bars->dsum, li & 1, abort_flag, kWaitBudget)) { ok = false; break; }
        const float d_exact = ds_item[row] + ds_item[kRows + row];
        corr = d_row - d_exact;
        if (g == 0 && grow < N) p.D[hb + grow] = live_row ? d_exact : 0.0f;
      }
      if constexpr (Cfg::kDefer) {
        epi_pend = true;
        ew_pend = w;
        eli_pend = li;
      } else if (!epilogue(w, li, corr)) {
        ok = false;
        break;
      }
      cbase += w.nb;
    }
    if (ok && Cfg::kDefer && epi_pend && !epilogue(ew_pend, eli_pend, 0.0f)) ok = false;
    if (!ok) raise_abort(bars, p.status);
    // the gradient stores must have completed before the CTA exits
    if (kWide && !kF32Grad && threadIdx.x == 128) {
      release_rows();
      bulk_wait_all();
    }
    __syncwarp();
  }
  };
  if (warp < 4) {
    regs_dec<kRegsHelper>();
    helper_roles();
  } else {
    regs_inc<kRegsElem>();
    elementwise_role();
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

template <int DP, bool kCausal, bool kDkDv, bool kF32, bool kF16>
cudaError_t launch_one(const BwdParams& p, cudaStream_t st) {
  using Cfg = BwdCfg<DP, kDkDv>;
  CUtensorMap m[7];
  // dQ:    rows are Q, dO (128-row boxes), blocks are K, V.
  // dK/dV: rows are K, V, blocks are Q, dO.
  const void* r1 = kDkDv ? p.k : p.q;
  const void* r2 = kDkDv ? p.v : p.dO;
  const void* c1 = kDkDv ? p.q : p.k;
  const void* c2 = kDkDv ? p.dO : p.v;
  cudaError_t e = make_bhnd_tmap(&m[0], r1, p.B, p.N, p.H, p.d, kRows, 64, kF16);
  if (e == cudaSuccess) e = make_bhnd_tmap(&m[1], r2, p.B, p.N, p.H, p.d, kRows, 64, kF16);
  if (e == cudaSuccess) e = make_bhnd_tmap(&m[2], c1, p.B, p.N, p.H, p.d, Cfg::kBlk, 64, kF16);
  if (e == cudaSuccess) e = make_bhnd_tmap(&m[3], c2, p.B, p.N, p.H, p.d, Cfg::kBlk, 64, kF16);
  // gradient outputs (bf16 gradients in the wide layout are stored by TMA):
  // dK/dV kernel: dV, dK; dQ kernel: dQ.  Unused otherwise (copies of m[0]).
  m[4] = m[0];
  m[5] = m[0];
  if (e == cudaSuccess && Cfg::kWide && !kF32) {
    e = make_bhnd_tmap(&m[4], kDkDv ? p.dv : p.dq, p.B, p.N, p.H, p.d, kRows, 64, kF16);
    if (e == cudaSuccess && kDkDv)
      e = make_bhnd_tmap(&m[5], p.dk, p.B, p.N, p.H, p.d, kRows, 64, kF16);
  }
  // the wide dQ kernel's O rows (it forms D's first estimate itself)
  m[6] = m[0];
  if (e == cudaSuccess && Cfg::kOwnD)
    e = make_bhnd_tmap(&m[6], p.o, p.B, p.N, p.H, p.d, kRows, 64, kF16);
  if (e != cudaSuccess) return e;
  auto kern = bwd_tc_kernel<DP, kCausal, kDkDv, kF32, kF16>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>((p.N + kRows - 1) / kRows) * p.B * p.H;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  BwdParams pc = p;
  void* args[] = {&m[0], &m[1], &m[2], &m[3], &m[4], &m[5], &m[6], &pc};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(kThreads), args,
                          Cfg::kSmemBytes, st);
}

// Phase 1 is the dQ kernel: it refines D in the workspace, which the dK/dV
// kernel (phase 2) then reads, so the phases run in that order.
template <int DP, bool kCausal, bool kF32>
cudaError_t launch_phase(const BwdParams& p, cudaStream_t st, int phase) {
  if (p.f16)
    return phase == 1 ? launch_one<DP, kCausal, false, kF32, true>(p, st)
                      : launch_one<DP, kCausal, true, kF32, true>(p, st);
  return phase == 1 ? launch_one<DP, kCausal, false, kF32, false>(p, st)
                    : launch_one<DP, kCausal, true, kF32, false>(p, st);
}

template <int DP>
cudaError_t launch_dp(const BwdParams& p, cudaStream_t st, bool causal, int phase) {
  if (causal) return p.grad_f32 ? launch_phase<DP, true, true>(p, st, phase)
                                : launch_phase<DP, true, false>(p, st, phase);
  return p.grad_f32 ? launch_phase<DP, false, true>(p, st, phase)
                    : launch_phase<DP, false, false>(p, st, phase);
}

}  // namespace

cudaError_t launch_bwd_tc16(const BwdParams& p, cudaStream_t s, bool causal, int phase) {
  if (phase != 1 && phase != 2) return cudaErrorInvalidValue;
  if (p.d <= 64) return launch_dp<64>(p, s, causal, phase);
  if (p.d <= 128) return launch_dp<128>(p, s, causal, phase);
  return cudaErrorNotSupported;
}

}  // namespace fa
