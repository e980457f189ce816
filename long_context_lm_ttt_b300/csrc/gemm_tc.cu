// gemm_tc.cu — persistent, warp-specialised bf16 GEMM on the 5th-generation
// tensor cores (tcgen05) with TMA-fed shared-memory pipelines and the fused
// epilogues of common.cuh.
//
//   C[m, n] = sum_k A(m, k) B(n, k)     (fp32 accumulate in TMEM)
//
// Tile 128 x BN x 64 (BN = 128 or 256).  Per CTA (one per SM, persistent
// over output tiles):
//   warp 0     TMA producer: A and B tiles into a STAGES-deep ring of
//              128-byte-swizzled shared-memory buffers (mbarrier full/empty);
//   warp 1     allocates TMEM (two BN-column fp32 accumulators) and issues
//              tcgen05.mma from one thread; tcgen05.commit frees smem stages
//              and publishes finished accumulators;
//   warps 2-5  epilogue: tcgen05.ld 32 columns at a time (each thread owns
//              one output row), apply the epilogue, release the accumulator,
//              so the next tile's MMAs overlap this tile's epilogue.
// Either operand may be K-major (rows of K contiguous) or MN-major (K rows of
// M/N contiguous); the TMA box orientation and the descriptor's major bit
// follow.  All waits are bounded (see tc_common.cuh).
#include <cuda.h>

#include <atomic>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace ttt {

namespace {

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;

// SRC = 1 (the SGD epilogue): the tile's fp32 master weights are brought
// into shared memory by TMA at the start of each tile, so the load overlaps
// the tile's main loop.  The epilogue updates them in place and writes the
// bf16 copy hi = rn(w) (and, when a low half is wanted, lo = rn(w - hi))
// into a staging tile; each epilogue warp then sends its 32 rows of the
// outputs back with TMA stores, so every global write is a whole 128-byte
// line.
//
// PAIR = 1: a cluster of two CTAs (on the two SMs of a TPC) computes a
// 256 x BN tile with tcgen05 MMAs of M = 256 (cta_group::2).  CTA r of the
// pair holds rows [128 r, 128 r + 128) of the A tile and columns
// [r BN/2, (r + 1) BN/2) of the B tile, and its TMEM receives rows
// [128 r, 128 r + 128) of the accumulator.  Each SM thus loads half of the
// B tile of a one-CTA 128 x BN tile, so a stage is smaller and the ring
// deeper in the same shared memory.
constexpr int kSmemMax = 232448;  // per-CTA opt-in limit
template <int BN, int SRC = 0, int PAIR = 0>
struct Cfg {
  static constexpr int BNL = PAIR ? BN / 2 : BN;  // B rows this CTA loads
  static constexpr int TM = PAIR ? 2 * BM : BM;   // rows of a work tile
  static constexpr int B_BYTES = BNL * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // SRC: the master tile moves through two slots of 64 columns (one slice
  // each, 32 KB fp32); the bf16 pair of the slice being stored is staged in
  // one 64-column slot of hi and one of lo (16 KB each)
  static constexpr int SLICES = BN / 64;
  static constexpr int SLOT_BYTES = BM * 64 * 4;
  static constexpr int SRC_BYTES = SRC ? 2 * SLOT_BYTES : 0;
  static constexpr int HL_BYTES = SRC ? 2 * BM * 128 : 0;
  static constexpr int FIT_STAGES = (kSmemMax - 2048 - SRC_BYTES - HL_BYTES) / STAGE_BYTES;
  static constexpr int STAGES =
      (PAIR || SRC) ? (FIT_STAGES > 8 ? 8 : FIT_STAGES) : (BN == 256 ? 4 : (BN == 192 ? 5 : 6));
  static constexpr int TMEM_COLS = 2 * BN;  // two accumulators
  // columns allocated: a power of two, at least 32
  static constexpr int TMEM_ALLOC = TMEM_COLS <= 32 ? 32 : TMEM_COLS <= 64 ? 64 : TMEM_COLS <= 128 ? 128
                                    : TMEM_COLS <= 256 ? 256 : 512;
  static constexpr int SRC_OFF = STAGES * STAGE_BYTES;
  static constexpr int HL_OFF = SRC_OFF + SRC_BYTES;
  static constexpr int BAR_OFF = HL_OFF + HL_BYTES;
  static constexpr int SMEM = 1024 /*align slack*/ + BAR_OFF + 256;
  static_assert(SMEM <= kSmemMax, "shared memory");
  static_assert(TMEM_COLS <= 512, "tensor memory");
  static_assert(BN % 32 == 0 && BNL % 8 == 0, "tile width");
  static_assert(8 * (2 * STAGES + 9) + 8 <= 256, "barrier area");
};

enum : int { ERR_WAIT_PRODUCER = 101, ERR_WAIT_MMA = 102, ERR_WAIT_EPI = 103, ERR_WAIT_DRAIN = 104 };

// Tile t -> (row tile, column tile) in groups of GROUP_M row tiles: inside a
// group the row index runs fastest, then the column index.  The tiles in
// flight at once (one per SM) then share GROUP_M row strips of A and a few
// column strips of B, which stay in L2, instead of streaming all of A once
// per column tile.
constexpr int GROUP_M = 16;
__device__ __forceinline__ void tile_mn(int t, int num_m, int num_n, int* mt, int* nt) {
  const int per_group = GROUP_M * num_n;
  const int g = t / per_group, r = t % per_group;
  const int first = g * GROUP_M;
  const int gm = min(num_m - first, GROUP_M);
  *mt = first + r % gm;
  *nt = r / gm;
}

template <int BN, int A_MN, int B_MN, int SRC = 0, int PAIR = 0>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapB2, const __grid_constant__ CUtensorMap mapS,
                   const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapH,
                   const __grid_constant__ CUtensorMap mapL, int dual, int M, int N, int K, Epi e, int* err,
                   int splits, float* ws, int grp_rows) {
  using C = Cfg<BN, SRC, PAIR>;
  // an MN-major B tile arrives in 64-column boxes
  static_assert(!B_MN || C::BNL % 64 == 0, "MN-major B needs whole 64-column boxes");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = tc::smem_u32(smem);
  uint64_t* bars = (uint64_t*)(smem + C::BAR_OFF);
  // bars: full[S], empty[S], tfull[2], tempty[2], drain
  const uint32_t full0 = tc::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * C::STAGES;
  const uint32_t tfull0 = empty0 + 8 * C::STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const uint32_t src_full = drain + 8;        // [2] halves of the master tile (SRC only)
  const uint32_t src_empty = src_full + 16;   // [2]
  uint32_t* tmem_slot = (uint32_t*)(smem + C::BAR_OFF + 8 * (2 * C::STAGES + 9));
  volatile int* abort = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work units go to CTAs, or with PAIR to CTA pairs (clusters of two)
  const int rank = PAIR ? (int)tc::cluster_rank() : 0;
  const int unit0 = PAIR ? (int)tc::cluster_id() : (int)blockIdx.x;
  const int ustride = PAIR ? (int)tc::cluster_count() : (int)gridDim.x;
  const int num_m = (M + C::TM - 1) / C::TM, num_n = (N + BN - 1) / BN;
  const int ntiles = num_m * num_n;
  const int nk = (K + BK - 1) / BK;
  const int nk_total = dual ? 2 * nk : nk;  // dual: A B^T then A B2^T into one accumulator
  // work units: (split, tile); split s covers k-blocks [kb_lo(s), kb_lo(s+1))
  const int nunits = ntiles * splits;
  auto kb_lo = [&](int sp) { return (int)((long long)sp * nk_total / splits); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      tc::mbar_init(full0 + 8 * s, 1);
      tc::mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(tfull0 + 8 * a, 1);
      // PAIR: one arrival per epilogue warp of both CTAs, on the first CTA's
      tc::mbar_init(tempty0 + 8 * a, PAIR ? 8 : 128);
    }
    tc::mbar_init(drain, 1);
    for (int j = 0; j < 2; ++j) {
      tc::mbar_init(src_full + 8 * j, 1);
      tc::mbar_init(src_empty + 8 * j, 4);  // one arrival per epilogue warp
    }
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&mapA);
    tc::prefetch_tmap(&mapB);
    if (dual) tc::prefetch_tmap(&mapB2);
    if (SRC) {
      tc::prefetch_tmap(&mapS);
      tc::prefetch_tmap(&mapW);
      tc::prefetch_tmap(&mapH);
      tc::prefetch_tmap(&mapL);
    }
  }
  if (warp == 1) {
    if (PAIR) {
      tc::tmem_alloc_pair(tc::smem_u32(tmem_slot), C::TMEM_ALLOC);
      tc::tmem_relinquish_pair();
    } else {
      tc::tmem_alloc(tc::smem_u32(tmem_slot), C::TMEM_ALLOC);
      tc::tmem_relinquish();
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  // PAIR: the peer's barriers must be initialised before the first remote
  // arrival or copy completion
  if (PAIR) tc::cluster_sync();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything below reads what earlier kernels wrote
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      int last_parity[C::STAGES];
      for (int s = 0; s < C::STAGES; ++s) last_parity[s] = -1;
      bool ok = true;
      // SRC: the 64-column slices of the master tiles of this CTA's units go,
      // in order, into the two slots as soon as the epilogue has stored a
      // slot's previous slice.  The producer issues them whenever it finds
      // a slot free, also while it waits for a pipeline stage, and waits
      // for slots only once every k-block has been issued, so the main loop
      // never waits for them.  gs counts slices issued.
      const int src_total = SRC && unit0 < nunits ? ((nunits - 1 - unit0) / ustride + 1) * C::SLICES : 0;
      int gs = 0;
      auto issue_src = [&] {
        const int u = unit0 + (gs / C::SLICES) * ustride, sl = gs % C::SLICES;
        int sm_, sn_;
        tile_mn(u % ntiles, num_m, num_n, &sm_, &sn_);
        const uint32_t sf = src_full + 8 * (gs & 1);
        tc::mbar_arrive_expect_tx(sf, C::SLOT_BYTES);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tc::tma_load_2d(sbase + C::SRC_OFF + (gs & 1) * C::SLOT_BYTES + j * BM * 128, &mapS,
                          sn_ * BN + 64 * sl + 32 * j, sm_ * C::TM + rank * BM, sf);
        ++gs;
      };
      auto slot_bar = [&] { return src_empty + 8 * (gs & 1); };
      auto slot_par = [&] { return (uint32_t)(((gs >> 1) & 1) ^ 1); };
      auto pump = [&] {
        while (gs < src_total && tc::mbar_try_wait(slot_bar(), slot_par())) issue_src();
      };
      // wait for a free pipeline stage (SRC: issuing slices meanwhile)
      auto wait_stage = [&](uint32_t bar, uint32_t par) -> bool {
        if (!SRC) return tc::mbar_wait(bar, par, err, ERR_WAIT_PRODUCER, abort);
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(bar, par)) {
          pump();
          if (*abort) return false;
          if (clock64() - t0 > tc::kWaitClocks) {
            atomicCAS(err, 0, ERR_WAIT_PRODUCER);
            *abort = 1;
            return false;
          }
        }
        return true;
      };
      int lu = 0;  // this CTA's unit counter
      for (int u = unit0; u < nunits && ok; u += ustride, ++lu) {
        const int t = u % ntiles, sp = u / ntiles;
        int mt_, nt_;
        tile_mn(t, num_m, num_n, &mt_, &nt_);
        // this CTA's rows of the tile and the B columns it loads
        const int m0 = mt_ * C::TM + rank * BM, n0 = nt_ * BN, nb0 = n0 + rank * C::BNL;
        for (int kb = kb_lo(sp); kb < kb_lo(sp + 1); ++kb) {
          if (SRC) pump();
          if (!wait_stage(empty0 + 8 * stage, phase ^ 1)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * stage;
          const uint32_t a_s = sbase + stage * C::STAGE_BYTES;
          const uint32_t b_s = a_s + A_BYTES;
          const int k0 = (kb < nk ? kb : kb - nk) * BK;
          const CUtensorMap* mb = kb < nk ? &mapB : &mapB2;
          if (PAIR) {
            // both halves of the stage complete on the first CTA's barrier,
            // which expects the bytes of both
            const uint32_t fbc = tc::mapa(fb, 0);
            if (rank == 0) tc::mbar_arrive_expect_tx(fb, 2 * C::STAGE_BYTES);
            if (A_MN) {
              tc::tma_load_2d_pair(a_s, &mapA, m0, k0, fbc);
              tc::tma_load_2d_pair(a_s + 8192, &mapA, m0 + 64, k0, fbc);
            } else {
              tc::tma_load_2d_pair(a_s, &mapA, k0, m0, fbc);
            }
            if (grp_rows) {
              // grouped: B of the tile's group through the 3-D map
              const int gi = mt_ * C::TM / grp_rows;
              if (B_MN) {
#pragma unroll
                for (int j = 0; j < C::BNL / 64; ++j)
                  tc::tma_load_3d_pair(b_s + 8192 * j, mb, nb0 + 64 * j, k0, gi, fbc);
              } else {
                tc::tma_load_3d_pair(b_s, mb, k0, nb0, gi, fbc);
              }
            } else if (B_MN) {
#pragma unroll
              for (int j = 0; j < C::BNL / 64; ++j) tc::tma_load_2d_pair(b_s + 8192 * j, mb, nb0 + 64 * j, k0, fbc);
            } else {
              tc::tma_load_2d_pair(b_s, mb, k0, nb0, fbc);
            }
          } else {
            tc::mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
            if (A_MN) {
              tc::tma_load_2d(a_s, &mapA, m0, k0, fb);
              tc::tma_load_2d(a_s + 8192, &mapA, m0 + 64, k0, fb);
            } else {
              tc::tma_load_2d(a_s, &mapA, k0, m0, fb);
            }
            if (grp_rows) {
              const int gi = mt_ * C::TM / grp_rows;
              if (B_MN) {
#pragma unroll
                for (int j = 0; j < BN / 64; ++j) tc::tma_load_3d(b_s + 8192 * j, mb, n0 + 64 * j, k0, gi, fb);
              } else {
                tc::tma_load_3d(b_s, mb, k0, n0, gi, fb);
              }
            } else if (B_MN) {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) tc::tma_load_2d(b_s + 8192 * j, mb, n0 + 64 * j, k0, fb);
            } else {
              tc::tma_load_2d(b_s, mb, k0, n0, fb);
            }
          }
          last_parity[stage] = (int)phase;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      while (ok && gs < src_total) {
        if (!tc::mbar_wait(slot_bar(), slot_par(), err, ERR_WAIT_PRODUCER, abort)) {
          ok = false;
          break;
        }
        issue_src();
      }
      if (!ok) {
        // let copies already issued land before the CTA exits (PAIR: the
        // second CTA's copies complete on the first CTA's barriers, which
        // it cannot poll, so it waits a fixed while instead)
        if (PAIR && rank != 0) {
          const long long t0 = clock64();
          while (clock64() - t0 < 4000000) {
          }
        } else {
          for (int s = 0; s < C::STAGES; ++s)
            if (last_parity[s] >= 0) {
              const long long t0 = clock64();
              while (!tc::mbar_try_wait(full0 + 8 * s, (uint32_t)last_parity[s]) &&
                     clock64() - t0 < tc::kWaitClocks) {
              }
            }
        }
        // and the last master-tile slice of each slot
        for (int k = gs > 2 ? gs - 2 : 0; k < gs; ++k) {
          const long long t0 = clock64();
          while (!tc::mbar_try_wait(src_full + 8 * (k & 1), (uint32_t)((k >> 1) & 1)) &&
                 clock64() - t0 < tc::kWaitClocks) {
          }
        }
      } else if (PAIR) {
        // the MMA issuer's releases of this CTA's stages arrive from the
        // other SM: wait for the last release of every stage before exit
        for (int i = 0; i < C::STAGES && ok; ++i) {
          ok = tc::mbar_wait(empty0 + 8 * stage, phase ^ 1, err, ERR_WAIT_PRODUCER, abort);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (PAIR: the first CTA's, for both) ----------------
      constexpr uint32_t idesc = tc::idesc_bf16(C::TM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued = false;
      for (int u = unit0; u < nunits && ok; u += ustride) {
        const int sp = u / ntiles;
        const int kb_first = kb_lo(sp);
        if (!tc::mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, err, ERR_WAIT_MMA, abort)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        for (int kb = kb_first; kb < kb_lo(sp + 1); ++kb) {
          if (!tc::mbar_wait(full0 + 8 * stage, phase, err, ERR_WAIT_MMA, abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a_s = sbase + stage * C::STAGE_BYTES;
          const uint32_t b_s = a_s + A_BYTES;
#pragma unroll
          for (int j = 0; j < BK / 16; ++j) {
            const uint64_t ad = A_MN ? tc::smem_desc_sw128(a_s + 2048 * j, 8192, 1024)
                                     : tc::smem_desc_sw128(a_s + 32 * j, 16, 1024);
            const uint64_t bd = B_MN ? tc::smem_desc_sw128(b_s + 2048 * j, 8192, 1024)
                                     : tc::smem_desc_sw128(b_s + 32 * j, 16, 1024);
            if (PAIR)
              tc::mma_bf16_pair(d_tmem, ad, bd, idesc, (kb != kb_first || j != 0) ? 1u : 0u);
            else
              tc::mma_bf16(d_tmem, ad, bd, idesc, (kb != kb_first || j != 0) ? 1u : 0u);
          }
          issued = true;
          if (PAIR)
            tc::mma_commit_pair(empty0 + 8 * stage, 3);
          else
            tc::mma_commit(empty0 + 8 * stage);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if (PAIR)
          tc::mma_commit_pair(tfull0 + 8 * acc, 3);
        else
          tc::mma_commit(tfull0 + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok && issued) {
        // drain MMAs in flight before TMEM is released
        if (PAIR)
          tc::mma_commit_pair(drain, 1);
        else
          tc::mma_commit(drain);
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(drain, 0) && clock64() - t0 < tc::kWaitClocks) {
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    // Thread i of a warp owns TMEM lane (tile row) i and applies the
    // epilogue to its row 32 columns at a time (epi_row32: 16-byte loads and
    // stores).  The source operand of the next chunk is loaded before the
    // current chunk is processed, the first chunk's before the accumulator
    // is waited for, so global-load latency overlaps useful work.
    // With split K the epilogue only stores the fp32 partial sum of its
    // split into ws[split][M][N]; splitk_reduce_kernel applies the epilogue.
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const bool partial = splits > 1;
    const bool has_src = !SRC && !partial && epi_has_src(e);
    const int trow = quarter * 32 + lane;  // row within the tile
    int acc = 0;
    uint32_t acc_phase = 0;
    int lu = 0;
    int gs = 0;  // SRC: master-tile slices consumed
    for (int u = unit0; u < nunits; u += ustride, ++lu) {
      const int t = u % ntiles, sp = u / ntiles;
      int mt_, nt_;
      tile_mn(t, num_m, num_n, &mt_, &nt_);
      const int m0 = mt_ * C::TM + rank * BM, n0 = nt_ * BN;
      const int row = m0 + trow;
      const int nch = min(BN, N - n0 + 31) / 32;  // chunks with columns < N
      auto vec_chunk = [&](int c) { return e.vec && n0 + 32 * c + 32 <= N; };
      uint4 src[8];
      if (has_src && row < M && vec_chunk(0)) epi_src_load(e, row, n0, src);
      if (!tc::mbar_wait(tfull0 + 8 * acc, acc_phase, err, ERR_WAIT_EPI, abort)) break;
      tc::tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      // release the accumulator once this warp's TMEM reads are done
      auto release_acc = [&] {
        tc::tc_fence_before();
        if (PAIR) {
          __syncwarp();
          if (lane == 0) tc::mbar_arrive_cluster(tc::mapa(tempty0 + 8 * acc, 0));
        } else {
          tc::mbar_arrive(tempty0 + 8 * acc);
        }
      };
      if (SRC) {
        // One 64-column slice at a time: w -= lr * acc on this row's bytes
        // of the slice's slot of the master tile (128-byte swizzle), in
        // place; hi = rn(w) and lo = rn(w - hi) into the staging slots
        // ([128 rows][128 B] each); then this warp's 32 rows of the slice go
        // out by TMA (boxes past the last row or column are not issued), and
        // the slots are released once the stores have read them.
        bool failed = false;
#pragma unroll 1
        for (int sl = 0; sl < C::SLICES; ++sl, ++gs) {
          const uint32_t slot = sbase + C::SRC_OFF + (gs & 1) * C::SLOT_BYTES;
          if (!tc::mbar_wait(src_full + 8 * (gs & 1), (gs >> 1) & 1, err, ERR_WAIT_EPI, abort)) {
            failed = true;
            break;
          }
#pragma unroll 1
          for (int j = 0; j < 2; ++j) {
            const int c = 2 * sl + j;
            if (n0 + 32 * c >= N) continue;
            float v[32];
            tc::tmem_ld32(tbase + c * 32, v);
            const uint32_t rb = slot + j * BM * 128 + trow * 128;
            uint32_t hl[16], ll[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t ad = rb + ((i ^ (trow & 7)) << 4);
              float w0, w1, w2, w3;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(w0), "=f"(w1), "=f"(w2), "=f"(w3)
                           : "r"(ad));
              w0 -= e.lr * v[4 * i];
              w1 -= e.lr * v[4 * i + 1];
              w2 -= e.lr * v[4 * i + 2];
              w3 -= e.lr * v[4 * i + 3];
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(ad), "f"(w0), "f"(w1), "f"(w2), "f"(w3)
                           : "memory");
              hl[2 * i] = bf2(w0, w1);
              hl[2 * i + 1] = bf2(w2, w3);
              const float2 h01 = unbf2(hl[2 * i]), h23 = unbf2(hl[2 * i + 1]);
              ll[2 * i] = bf2(w0 - h01.x, w1 - h01.y);
              ll[2 * i + 1] = bf2(w2 - h23.x, w3 - h23.y);
            }
            const uint32_t hb = sbase + C::HL_OFF + trow * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t off = (((4 * j + i) ^ (trow & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(hb + off), "r"(hl[4 * i]),
                           "r"(hl[4 * i + 1]), "r"(hl[4 * i + 2]), "r"(hl[4 * i + 3])
                           : "memory");
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(hb + BM * 128 + off), "r"(ll[4 * i]),
                           "r"(ll[4 * i + 1]), "r"(ll[4 * i + 2]), "r"(ll[4 * i + 3])
                           : "memory");
            }
          }
          if (sl == C::SLICES - 1) release_acc();
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int r = m0 + quarter * 32, c0 = n0 + 64 * sl;
            if (r < M && c0 < N) {
              for (int j = 0; j < 2; ++j)
                if (c0 + 32 * j < N) tc::tma_store_2d(&mapW, c0 + 32 * j, r, slot + j * BM * 128 + quarter * 4096);
              const uint32_t hb = sbase + C::HL_OFF + quarter * 4096;
              tc::tma_store_2d(&mapH, c0, r, hb);
              if (e.w16lo) tc::tma_store_2d(&mapL, c0, r, hb + BM * 128);
            }
            tc::bulk_commit();
            tc::bulk_wait_read();
            tc::mbar_arrive(src_empty + 8 * (gs & 1));
          }
          __syncwarp();
        }
        if (failed) break;
      } else {
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          float v[32];
          tc::tmem_ld32(tbase + c * 32, v);
          uint4 nxt[8];
          if (has_src && row < M && c + 1 < nch && vec_chunk(c + 1)) epi_src_load(e, row, n0 + 32 * (c + 1), nxt);
          if (row < M && partial) {
            float* wp = ws + ((int64_t)sp * M + row) * N + n0 + 32 * c;
            if (vec_chunk(c) && (N & 3) == 0) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                stg16(wp + 4 * i, make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                                             __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3])));
            } else {
#pragma unroll
              for (int k = 0; k < 32; ++k)
                if (n0 + 32 * c + k < N) wp[k] = v[k];
            }
          } else if (row < M) {
            if (vec_chunk(c)) {
              epi_row32(e, row, n0 + 32 * c, v, src);
            } else {
#pragma unroll
              for (int p = 0; p < 16; ++p) {
                const int col = n0 + c * 32 + 2 * p;
                if (col < N) epi_pair<bf16>(e, row, col, v[2 * p], v[2 * p + 1]);
              }
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) src[i] = nxt[i];
        }
        release_acc();
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    // global writes of the last stores complete before the CTA exits
    if (SRC && lane == 0) tc::bulk_wait_all();
  }
  tc::tc_fence_before();
  __syncthreads();
  // PAIR: neither CTA leaves (or frees TMEM) while the other may still
  // touch its barriers or write its accumulator
  if (PAIR) tc::cluster_sync();
  if (warp == 1) {
    tc::tc_fence_after();
    if (PAIR)
      tc::tmem_dealloc_pair(tmem, C::TMEM_ALLOC);
    else
      tc::tmem_dealloc(tmem, C::TMEM_ALLOC);
  }
}

// Sum of the split-K partials (fixed order) through the epilogue; one thread
// per (row, 32-column chunk), consecutive threads on consecutive chunks.
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, int splits, int M, int N, Epi e) {
  pdl_wait();
  pdl_trigger();
  const int nch = (N + 31) / 32;
  const int64_t total = (int64_t)M * nch;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int row = (int)(i / nch), col0 = (int)(i % nch) * 32;
    const bool vec = e.vec && col0 + 32 <= N && (N & 3) == 0;
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = 0.f;
    for (int sp = 0; sp < splits; ++sp) {
      const float* p = ws + ((int64_t)sp * M + row) * N + col0;
      if (vec) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 x = *reinterpret_cast<const float4*>(p + 4 * q);
          v[4 * q] += x.x;
          v[4 * q + 1] += x.y;
          v[4 * q + 2] += x.z;
          v[4 * q + 3] += x.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (col0 + k < N) v[k] += p[k];
      }
    }
    if (vec) {
      uint4 src[8];
      if (epi_has_src(e)) epi_src_load(e, row, col0, src);
      epi_row32(e, row, col0, v, src);
    } else {
#pragma unroll
      for (int p = 0; p < 16; ++p)
        if (col0 + 2 * p < N) epi_pair<bf16>(e, row, col0 + 2 * p, v[2 * p], v[2 * p + 1]);
    }
  }
}

// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
int g_init_rc = 0;

int make_map(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld_elems,
             uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld_elems * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

// bf16 3-D map: `groups` matrices of [outer, inner] (pitch ld_elems), each
// group_stride elements after the previous; box {64, box_outer, 1}
int make_map3(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld_elems, uint64_t groups,
              uint64_t group_stride, uint32_t box_outer) {
  cuuint64_t dims[3] = {inner, outer, groups};
  cuuint64_t strides[2] = {ld_elems * 2, group_stride * 2};
  cuuint32_t box[3] = {64, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

// fp32 [rows, cols] tile map with 128-byte swizzle: box {32 columns, box_rows}
int make_map_f32(CUtensorMap* map, const void* ptr, uint64_t cols, uint64_t rows, uint64_t ld_elems,
                 uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld_elems * 4};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

template <int BN, int A_MN, int B_MN, int SRC = 0, int PAIR = 0>
int launch(const GemmArgs<bf16>& g, int num_sms, int* err, cudaStream_t st, int splits) {
  using C = Cfg<BN, SRC, PAIR>;
  CUtensorMap ma, mb, mb2, ms, mw, mh, ml;
  int rc;
  if (A_MN) rc = make_map(&ma, g.A, g.M, g.K, g.lda, 64, 64);
  else rc = make_map(&ma, g.A, g.K, g.M, g.lda, 64, BM);
  if (rc) return rc;
  const bool grouped = g.groups > 1;
  auto map_b = [&](CUtensorMap* m, const bf16* ptr) {
    if (grouped)
      return B_MN ? make_map3(m, ptr, g.N, g.K, g.ldb, g.groups, g.group_stride, 64)
                  : make_map3(m, ptr, g.K, g.N, g.ldb, g.groups, g.group_stride, C::BNL);
    return B_MN ? make_map(m, ptr, g.N, g.K, g.ldb, 64, 64) : make_map(m, ptr, g.K, g.N, g.ldb, 64, C::BNL);
  };
  rc = map_b(&mb, g.B);
  if (rc) return rc;
  if (g.B2) {
    rc = map_b(&mb2, g.B2);
    if (rc) return rc;
  } else {
    mb2 = mb;
  }
  if (SRC) {
    // master tile in (128 rows), master / hi / lo out (32-row slab per warp)
    rc = make_map_f32(&ms, g.e.w32, g.N, g.M, g.e.ldo, BM);
    if (!rc) rc = make_map_f32(&mw, g.e.w32, g.N, g.M, g.e.ldo, 32);
    if (!rc) rc = make_map(&mh, g.e.w16, g.N, g.M, g.e.ldo, 64, 32);
    // no low half: the epilogue stores only w32 and w16
    if (!rc) {
      if (g.e.w16lo) rc = make_map(&ml, g.e.w16lo, g.N, g.M, g.e.ldo, 64, 32);
      else ml = mh;
    }
    if (rc) return rc;
  } else {
    ms = mw = mh = ml = mb;
  }
  auto kern = gemm_tc_kernel<BN, A_MN, B_MN, SRC, PAIR>;
  static std::atomic<uint64_t> attr_set{0};  // per instantiation, per device
  {
    cudaError_t e = raise_smem_limit(attr_set, kern, C::SMEM);
    if (e != cudaSuccess) return (int)e;
  }
  const int ntiles = ((g.M + C::TM - 1) / C::TM) * ((g.N + BN - 1) / BN);
  const int nunits = ntiles * splits;
  const int cap = g.grid_cap > 0 ? g.grid_cap : num_sms;
  if (PAIR) {
    // one unit per cluster of two CTAs, at most as many clusters as fit at once
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    static std::atomic<int> resident{0};  // per instantiation
    if (!resident) {
      cfg.gridDim = dim3(2 * (num_sms / 2));
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = num_sms / 2;
      }
      resident = n;
    }
    const int pairs = std::max(1, std::min(cap / 2, resident.load()));
    cfg.gridDim = dim3(2 * (nunits < pairs ? nunits : pairs));
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, kern, ma, mb, mb2, ms, mw, mh, ml, g.B2 ? 1 : 0, g.M, g.N, g.K,
                                              g.e, err, splits, g.ws, grouped ? g.group_rows : 0);
    if (le != cudaSuccess) return (int)le;
  } else {
    const int grid = nunits < cap ? nunits : cap;
    launch_k(kern, grid, 192, C::SMEM, st, ma, mb, mb2, ms, mw, mh, ml, g.B2 ? 1 : 0, g.M, g.N, g.K, g.e, err, splits,
                                     g.ws, grouped ? g.group_rows : 0);
  }
  if (splits > 1) {
    const int64_t items = (int64_t)g.M * ((g.N + 31) / 32);
    const int rgrid = (int)std::min<int64_t>((items + 127) / 128, (int64_t)num_sms * 16);
    launch_k(splitk_reduce_kernel, rgrid, 128, 0, st, g.ws, splits, g.M, g.N, g.e);
  }
  return (int)cudaPeekAtLastError();
}

template <int BN, int PAIR>
int dispatch_major(const GemmArgs<bf16>& g, int num_sms, int* err, cudaStream_t st, int splits) {
  if (g.a_mn) {
    return g.b_mn ? launch<BN, 1, 1, 0, PAIR>(g, num_sms, err, st, splits)
                  : launch<BN, 1, 0, 0, PAIR>(g, num_sms, err, st, splits);
  }
  return g.b_mn ? launch<BN, 0, 1, 0, PAIR>(g, num_sms, err, st, splits)
                : launch<BN, 0, 0, 0, PAIR>(g, num_sms, err, st, splits);
}
// 192-column tiles on CTA pairs: each CTA loads 96 rows of B, which only a
// K-major B provides in one box (the planner never picks it otherwise)
int dispatch_192_pair(const GemmArgs<bf16>& g, int num_sms, int* err, cudaStream_t st, int splits) {
  if (g.b_mn) return (int)cudaErrorNotSupported;
  return g.a_mn ? launch<192, 1, 0, 0, 1>(g, num_sms, err, st, splits)
                : launch<192, 0, 0, 0, 1>(g, num_sms, err, st, splits);
}

// Tile shape and K split by a simple time model: a k-block of a 128 x BN
// tile costs BN units (narrower tiles a little more per column: they are
// closer to the shared-memory bandwidth limit), tiles run in waves of
// num_sms, and a split adds a reduction pass over splits x M x N fp32.  A
// CTA pair runs a 256 x BN tile in the time a single CTA runs 128 x BN, in
// waves of num_sms / 2, and loads half as much B per SM (kPairGain).
// BN = 192 exists for outputs 3072 wide at M = 1024 (the chunk's o-proj,
// down-proj and most input-gradient products): 16 column tiles make 64 pair
// tiles (or 128 single ones), 86% of one wave, where 256-wide tiles leave
// 35% of the SMs idle.
struct Plan {
  int bn, splits, pair;
};
constexpr double kPairGain = 0.88;
static Plan plan_gemm(const GemmArgs<bf16>& g, int num_sms) {
  const int nk = (g.K + BK - 1) / BK;
  const int nkt = g.B2 ? 2 * nk : nk;
  // cost unit: one k-block of a 128 x 256 tile (~0.27 us at full rate)
  const double kb_us = 0.27;
  Plan best{128, 1, 0};
  double best_cost = 1e300;
  for (int pair = 0; pair <= 1; ++pair) {
    if (g.pair >= 0 ? pair != g.pair : (pair && g.M <= BM)) continue;
    const int slots = pair ? num_sms / 2 : num_sms;
    const int num_m = (g.M + (pair ? 2 * BM : BM) - 1) / (pair ? 2 * BM : BM);
    // on near-ties (3%) the earlier candidate stays: 192-wide tiles cost a
    // little more per column, so they come last and win only where they
    // fill a wave clearly better
    for (int bn : {128, 256, 192}) {
      if (bn > 128 && g.N <= 128) continue;
      if (bn == 192 && pair && g.b_mn) continue;  // see dispatch_192_pair
      const int tiles = num_m * ((g.N + bn - 1) / bn);
      const double kb_cost = (bn == 256 ? 1.0 : (bn == 192 ? 0.79 : 0.58)) * (pair ? kPairGain : 1.0) * kb_us;
      for (int sp = 1; sp <= 4; ++sp) {
        if (sp > 1 && (!g.ws || nkt / sp < 8 || (int64_t)sp * g.M * g.N > g.ws_elems)) break;
        const double waves = std::ceil((double)tiles * sp / slots);
        const int kb_unit = (nkt + sp - 1) / sp;
        double cost = waves * kb_unit * kb_cost;
        if (sp > 1) cost += 3.0 + (double)sp * g.M * g.N * 8.0 / 8e6;  // launch + L2-resident traffic (us)
        if (cost < best_cost * 0.97) {
          best_cost = cost;
          best = {bn, sp, pair};
        }
      }
    }
  }
  return best;
}

}  // namespace

int gemm_tc_init() {
  std::call_once(g_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
      g_init_rc = (int)cudaErrorNotSupported;
      return;
    }
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  });
  return g_init_rc;
}

// may the epilogue of g use 16-byte vector accesses (epi_row32)?
static bool a16(const void* p) { return ((uintptr_t)p & 15) == 0; }
static bool epi_vec_ok(const Epi& e) {
  const int64_t o4 = e.ldo * 4, o2 = e.ldo * 2;
  switch (e.kind) {
    case EPI_STORE: return a16(e.out) && ((e.out_f32 ? o4 : o2) % 16 == 0);
    case EPI_RESID: return a16(e.out) && a16(e.resid) && o4 % 16 == 0 && (e.ldr * 4) % 16 == 0;
    case EPI_QKV:
      return e.hd % 32 == 0 && a16(e.out) && a16(e.kring) && a16(e.vring) && a16(e.rope_cs) && o2 % 16 == 0;
    case EPI_SWIGLU:
      return a16(e.out) && o2 % 16 == 0 && (!e.stash || (a16(e.stash) && (e.ld_stash * 2) % 16 == 0));
    case EPI_SWIGLU_BWD: return a16(e.out) && a16(e.stash) && o2 % 16 == 0 && (e.ld_stash * 2) % 16 == 0;
    case EPI_SGD:
      return a16(e.w32) && o4 % 16 == 0 && (!e.w16 || a16(e.w16)) && (!e.w16lo || a16(e.w16lo));
    case EPI_CE_Z:
    case EPI_CE_ACC: return a16(e.out) && o4 % 16 == 0;
    default: return false;
  }
}

int gemm_tc(const GemmArgs<bf16>& g_in, int num_sms, int* err, cudaStream_t st, int* kernels) {
  GemmArgs<bf16> g = g_in;
  if (kernels) *kernels = 1;
  if (g.groups > 1) {
    // one launch for every group when whole tiles fall in one group (the
    // tile height divides group_rows; pairs need 256); otherwise one
    // launch per group
    const bool rows_ok = g.group_rows > 0 && (int64_t)g.groups * g.group_rows == g.M && g.e.kind != EPI_SGD;
    if (rows_ok && g.group_rows % BM == 0) {
      if (g.group_rows % (2 * BM) != 0) g.pair = 0;
    } else {
      int total = 0;
      for (int gi = 0; gi < g.groups; ++gi) {
        GemmArgs<bf16> s = g;
        const int64_t r0 = (int64_t)gi * g.group_rows;
        s.M = std::min<int64_t>(g.group_rows, g.M - r0);
        if (s.M <= 0) break;
        s.A = g.a_mn ? g.A + r0 : g.A + r0 * g.lda;
        s.B = g.B + gi * g.group_stride;
        s.B2 = g.B2 ? g.B2 + gi * g.group_stride : nullptr;
        s.e = epi_rows_from<bf16>(g.e, r0);
        s.groups = 1;
        s.group_rows = 0;
        int nk = 1;
        const int rc = gemm_tc(s, num_sms, err, st, &nk);
        if (rc) return rc;
        total += nk;
      }
      if (kernels) *kernels = total;
      return 0;
    }
  }
  g.e.vec = epi_vec_ok(g.e) ? 1 : 0;
  if (g.M <= 0 || g.N <= 0) return 0;
  // one row, K-major operands, 16-byte aligned rows: stream B once (gemv.cu)
  if (gemv_supported(g)) {
    gemv_row(g, num_sms, st);
    return (int)cudaPeekAtLastError();
  }
  if (!g_encode) return (int)cudaErrorNotSupported;
  // TMA: 16-byte aligned base and row pitch
  if (((uintptr_t)g.A & 15) || ((uintptr_t)g.B & 15) || ((uintptr_t)g.B2 & 15) || (g.lda & 7) ||
      (g.ldb & 7) || g.K <= 0)
    return (int)cudaErrorNotSupported;
  // the SGD epilogue (weight-gradient GEMM, both operands MN-major, a bf16
  // copy wanted, with or without its low half) updates the fp32 masters in
  // a TMA-fed shared-memory tile and stores the outputs by TMA
  if (g.e.kind == EPI_SGD && g.groups == 1 && g.e.vec && g.a_mn && g.b_mn && !g.B2 && (g.N % 32) == 0 && g.e.w16 &&
      (g.e.ldo % 8) == 0 && a16(g.e.w16) && (!g.e.w16lo || a16(g.e.w16lo))) {
    if (kernels) *kernels = 1;
    const bool pair = g.pair >= 0 ? g.pair == 1 : g.M > BM;
    return pair ? launch<256, 1, 1, 1, 1>(g, num_sms, err, st, 1) : launch<128, 1, 1, 1, 0>(g, num_sms, err, st, 1);
  }
  const Plan pl = plan_gemm(g, num_sms);
  if (pl.splits > 1 && (((uintptr_t)g.ws & 15) != 0)) return (int)cudaErrorNotSupported;
  if (kernels) *kernels = pl.splits > 1 ? 2 : 1;
  if (pl.pair) {
    if (pl.bn == 192) return dispatch_192_pair(g, num_sms, err, st, pl.splits);
    return pl.bn == 256 ? dispatch_major<256, 1>(g, num_sms, err, st, pl.splits)
                        : dispatch_major<128, 1>(g, num_sms, err, st, pl.splits);
  }
  if (pl.bn == 192) return dispatch_major<192, 0>(g, num_sms, err, st, pl.splits);
  return pl.bn == 256 ? dispatch_major<256, 0>(g, num_sms, err, st, pl.splits)
                      : dispatch_major<128, 0>(g, num_sms, err, st, pl.splits);
}

}  // namespace ttt
