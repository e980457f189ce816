// attn_tc.cu — sliding-window causal attention on the 5th-generation tensor
// cores (tcgen05), forward and chunk-local backward, bf16 in / fp32 math.
//
// Geometry shared by every kernel here:
//   * a query tile is 128 consecutive rows of the chunk (one TMEM lane per
//     row); a key block is BN = 64 consecutive absolute positions starting
//     at a multiple of 64, so its ring slots (p mod R, R a multiple of 128)
//     are contiguous and one TMA box fetches it;
//   * query t (absolute) sees keys j with t - W < j <= t; key blocks that
//     straddle either edge are masked element-wise, interior blocks are not;
//   * head_dim hd <= 128 is split into 64-wide "atoms" of 128 bytes, the
//     unit of the 128-byte swizzle shared by TMA and the MMA descriptors.
//     With hd = 96 the second atom's upper half is zero (key/value maps end
//     at hd) or ignored (q/o/dO rows: the MMA reads hd/16 K-steps only).
//
// Forward, one CTA per (query tile, head), 6 warps:
//   warp 0    TMA producer: Q once, then K and V blocks into a 2-stage ring;
//   warp 1    TMEM owner and MMA issuer: S_i = Q K_i^T into one of two
//             64-column TMEM buffers, then O += P_i V_i (O in TMEM);
//   warps 2-5 softmax, one query row per thread: read S_i, mask, online
//             max with lazy rescaling of O (only when the running max grows
//             by more than 2^8), write P_i (bf16) into shared memory in the
//             swizzled K-major layout the MMA reads, and at the end scale O
//             by 1/l and store it with the row's log-sum-exp.
// S_{i+1} is issued before P_i V_i so the tensor core works on the next
// scores while the softmax warps work on the current ones.  Two CTAs fit on
// one SM (112 KB shared memory, 256 TMEM columns each).
#include <cuda.h>

#include <atomic>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "bounds.cuh"
#include "tc_common.cuh"

namespace ttt {

TTT_BOUNDS_UNIT(attn_tc)

namespace {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 64;    // keys per block
constexpr int STAGES = 2; // key/value ring depth

enum : int {
  ERR_A_PROD = 201,
  ERR_A_MMA = 202,
  ERR_A_SOFT = 203,
};

// shared-memory map of the forward kernel for NA head-dim atoms
template <int NA>
struct FwdSmem {
  static constexpr int Q_BYTES = NA * BM * 128;
  static constexpr int KV_BYTES = NA * BN * 128;
  static constexpr int P_BYTES = BM * BN * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + Q_BYTES;
  static constexpr int V_OFF = K_OFF + STAGES * KV_BYTES;
  static constexpr int P_OFF = V_OFF + STAGES * KV_BYTES;
  static constexpr int BAR_OFF = P_OFF + P_BYTES;
  // at least 80 KB so that no more than two CTAs (2 x 256 TMEM columns)
  // share an SM
  static constexpr int SMEM = BAR_OFF + 256 > 80 * 1024 ? BAR_OFF + 256 : 80 * 1024;
};

struct FwdParams {
  int n, H, Hkv, hd, W, R;
  long long pos0;
  float scale_log2;  // log2(e) / sqrt(hd)
  bf16* o;
  int64_t ldo;
  float* lse;
  int ld_lse;
  int* err;
  // two-tile kernel with the key range split into parts (parts > 1): part
  // z leaves its unnormalised output in ws[z][row][H*hd] and its row
  // statistics (max in log2 units, sum) in ws_ml[z][h][row][2]; a combine
  // kernel merges the parts
  int parts;
  float* ws;
  float* ws_ml;
};

// first key block and block count of the query tile starting at row r0
__device__ __forceinline__ void tile_blocks(const FwdParams& p, int r0, long long* kb0, int* nb) {
  const long long t_lo = p.pos0 + r0;
  const long long t_hi = p.pos0 + min(r0 + BM, p.n) - 1;
  long long k_lo = t_lo - p.W + 1;
  if (k_lo < 0) k_lo = 0;
  *kb0 = k_lo / BN;
  *nb = (int)(t_hi / BN - *kb0 + 1);
}

// One arrival per warp on a hand-off barrier: every lane has finished (and
// fenced) its own shared/tensor-memory writes; the warp synchronises and
// lane 0 arrives, so the barrier counts warps rather than threads.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) tc::mbar_arrive(bar);
}

// every lane waits on the barrier; the warp agrees on the outcome so that
// warp-collective tcgen05 instructions are reached by all lanes or none
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* err, int code,
                                          volatile int* abort) {
  const bool ok = tc::mbar_wait(bar, parity, err, code, abort);
  return __all_sync(0xffffffffu, ok);
}

// A 2-D tile copy of a box of 64 bf16 columns and box_rows rows at column x,
// row y of a map of inner x outer elements.  The debug build checks that x
// lies on a 16-byte boundary (an unaligned start raises an illegal-
// instruction fault) and that the box starts inside the map's columns (its
// columns may run past the inner extent: head dims below 128 read zeros
// there).  Query and gradient boxes (ring = 0) may start past the last row:
// a tile pair whose second tile has no rows loads zeros.  A key/value box
// (ring > 0) must start inside the map and stay inside one head's ring of
// `ring` rows.  A failed check skips the copy and raises the kernel's abort
// flag, so every role leaves its bounded wait.
__device__ __forceinline__ void tma_load_box(int kid, uint32_t dst, const CUtensorMap* map, int x, int y, int inner,
                                             int outer, int box_rows, int ring, uint32_t bar, volatile int* abort) {
  if (TTT_IN(kid, x & 7, 1) && TTT_IN(kid, x, inner) &&
      (ring <= 0 || (TTT_IN(kid, y, outer) && TTT_IN(kid, y % ring + box_rows - 1, ring)))) {
    tc::tma_load_2d(dst, map, x, y, bar);
  } else {
    *abort = 1;
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// one row of 64 bf16 values into a 128-byte-swizzled K-major tile
__device__ __forceinline__ void store_row_sw128(uint32_t tile, int row, const float (&p)[64]) {
  const uint32_t base = tile + row * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t addr = base + ((c ^ (row & 7)) << 4);
    st_shared_v4(addr, pack_bf16(p[8 * c + 0], p[8 * c + 1]), pack_bf16(p[8 * c + 2], p[8 * c + 3]),
                 pack_bf16(p[8 * c + 4], p[8 * c + 5]), pack_bf16(p[8 * c + 6], p[8 * c + 7]));
  }
}

template <int NA>
__global__ void __launch_bounds__(192, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                       const __grid_constant__ CUtensorMap mapV, FwdParams p) {
  using SM = FwdSmem<NA>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + SM::BAR_OFF;
  // barriers (8 bytes each)
  const uint32_t q_full = bar0;
  const uint32_t k_full = bar0 + 8;          // [2]
  const uint32_t v_full = bar0 + 24;         // [2]
  const uint32_t kv_empty = bar0 + 40;       // [2]
  const uint32_t s_full = bar0 + 56;         // [2]
  const uint32_t s_empty = bar0 + 72;        // [2]
  const uint32_t p_full = bar0 + 88;
  const uint32_t o_done = bar0 + 96;
  uint32_t* tmem_slot = (uint32_t*)(smem + SM::BAR_OFF + 128);
  volatile int* abort = (volatile int*)(smem + SM::BAR_OFF + 132);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y;
  const int r0 = qt * BM;
  const int kvh = h / (p.H / p.Hkv);
  long long kb0;
  int nb;
  tile_blocks(p, r0, &kb0, &nb);
  const int ksteps = p.hd / 16;
  const int nO = (p.hd + 15) & ~15;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(k_full + 8 * s, 1);
      tc::mbar_init(v_full + 8 * s, 1);
      tc::mbar_init(kv_empty + 8 * s, 1);
      tc::mbar_init(s_full + 8 * s, 1);
      tc::mbar_init(s_empty + 8 * s, 128);
    }
    tc::mbar_init(p_full, 128);
    tc::mbar_init(o_done, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&mapQ);
    tc::prefetch_tmap(&mapK);
    tc::prefetch_tmap(&mapV);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), 256);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything below reads what earlier kernels wrote
  pdl_wait();
  pdl_trigger();
  const uint32_t tS = tmem;          // two 64-column score buffers
  const uint32_t tO = tmem + 128;    // output accumulator (nO columns)

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      bool ok = true;
      int issued = 0;
      tc::mbar_arrive_expect_tx(q_full, SM::Q_BYTES);
      for (int a = 0; a < NA; ++a)
        tma_load_box(KB_ATTN_FWD_TC, sbase + SM::Q_OFF + a * BM * 128, &mapQ, h * p.hd + 64 * a, r0,
                     p.H * p.hd, p.n, BM, 0, q_full, abort);
      for (int i = 0; i < nb && ok; ++i) {
        const int st = i & 1;
        if (!tc::mbar_wait(kv_empty + 8 * st, ((i >> 1) & 1) ^ 1, p.err, ERR_A_PROD, abort)) {
          ok = false;
          break;
        }
        const long long kpos = (kb0 + i) * BN;
        const int row = kvh * p.R + (int)(kpos % p.R);
        tc::mbar_arrive_expect_tx(k_full + 8 * st, SM::KV_BYTES);
        for (int a = 0; a < NA; ++a)
          tma_load_box(KB_ATTN_FWD_TC, sbase + SM::K_OFF + st * SM::KV_BYTES + a * BN * 128, &mapK, 64 * a, row,
                       p.hd, p.Hkv * p.R, BN, p.R, k_full + 8 * st, abort);
        tc::mbar_arrive_expect_tx(v_full + 8 * st, SM::KV_BYTES);
        for (int a = 0; a < NA; ++a)
          tma_load_box(KB_ATTN_FWD_TC, sbase + SM::V_OFF + st * SM::KV_BYTES + a * BN * 128, &mapV, 64 * a, row,
                       p.hd, p.Hkv * p.R, BN, p.R, v_full + 8 * st, abort);
        issued = i + 1;
      }
      // let copies in flight land before the CTA can exit
      const long long t0 = clock64();
      while (!tc::mbar_try_wait(q_full, 0) && clock64() - t0 < tc::kWaitClocks) {
      }
      for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i) {
        const int st = i & 1;
        const uint32_t par = (i >> 1) & 1;
        const long long t1 = clock64();
        while (!(tc::mbar_try_wait(k_full + 8 * st, par) && tc::mbar_try_wait(v_full + 8 * st, par)) &&
               clock64() - t1 < tc::kWaitClocks) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idS = tc::idesc_bf16(BM, BN, 0, 0);
      const uint32_t idO = tc::idesc_bf16(BM, nO, 0, 1);
      bool ok = tc::mbar_wait(q_full, 0, p.err, ERR_A_MMA, abort);
      bool issued = false;
      for (int i = 0; i <= nb && ok; ++i) {
        if (i < nb) {
          const int st = i & 1;
          const uint32_t par = (i >> 1) & 1;
          if (!tc::mbar_wait(k_full + 8 * st, par, p.err, ERR_A_MMA, abort) ||
              !tc::mbar_wait(s_empty + 8 * st, par ^ 1, p.err, ERR_A_MMA, abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t kb = sbase + SM::K_OFF + st * SM::KV_BYTES;
          for (int j = 0; j < ksteps; ++j) {
            const int a = j >> 2;
            const uint64_t ad = tc::smem_desc_sw128(sbase + SM::Q_OFF + a * BM * 128 + 32 * (j & 3), 16, 1024);
            const uint64_t bd = tc::smem_desc_sw128(kb + a * BN * 128 + 32 * (j & 3), 16, 1024);
            tc::mma_bf16(tS + st * BN, ad, bd, idS, j > 0);
          }
          issued = true;
          tc::mma_commit(s_full + 8 * st);
        }
        if (i >= 1) {
          const int k = i - 1;
          const int st = k & 1;
          if (!tc::mbar_wait(v_full + 8 * st, (k >> 1) & 1, p.err, ERR_A_MMA, abort) ||
              !tc::mbar_wait(p_full, k & 1, p.err, ERR_A_MMA, abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t vb = sbase + SM::V_OFF + st * SM::KV_BYTES;
#pragma unroll
          for (int j = 0; j < BN / 16; ++j) {
            const uint64_t ad = tc::smem_desc_sw128(sbase + SM::P_OFF + 32 * j, 16, 1024);
            const uint64_t bd = tc::smem_desc_sw128(vb + 2048 * j, BN * 128, 1024);
            tc::mma_bf16(tO, ad, bd, idO, (k > 0 || j > 0) ? 1u : 0u);
          }
          tc::mma_commit(o_done);
          tc::mma_commit(kv_empty + 8 * st);
        }
      }
      if (!ok && issued) {
        // drain MMAs in flight before TMEM is released
        const uint32_t drain = bar0 + 104;
        tc::mbar_init(drain, 1);
        tc::fence_mbar_init();
        tc::mma_commit(drain);
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(drain, 0) && clock64() - t0 < tc::kWaitClocks) {
        }
      }
    }
  } else {
    // ---------------- softmax (warps 2..5) ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;           // TMEM lane / tile row
    const long long t = p.pos0 + r0 + row;         // absolute position
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float NEG_INF = -INFINITY;
    float m_run = NEG_INF, l_run = 0.f;
    bool ok = true;
    for (int i = 0; i < nb; ++i) {
      const int st = i & 1;
      if (!warp_wait(s_full + 8 * st, (i >> 1) & 1, p.err, ERR_A_SOFT, abort)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      float s[64];
      {
        float (&s0)[32] = *reinterpret_cast<float(*)[32]>(&s[0]);
        float (&s1)[32] = *reinterpret_cast<float(*)[32]>(&s[32]);
        tc::tmem_ld32(tS + st * BN + lane_off, s0);
        tc::tmem_ld32(tS + st * BN + 32 + lane_off, s1);
      }
      tc::tc_fence_before();
      tc::mbar_arrive(s_empty + 8 * st);
      // valid columns c: t - W < kpos + c <= t
      const long long kpos = (kb0 + i) * BN;
      const long long lo = t - p.W + 1 - kpos, hi = t - kpos;
      float mb = NEG_INF;
      if (lo <= 0 && hi >= BN - 1) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          s[c] *= p.scale_log2;
          mb = fmaxf(mb, s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          s[c] = (c >= lo && c <= hi) ? s[c] * p.scale_log2 : NEG_INF;
          mb = fmaxf(mb, s[c]);
        }
      }
      // lazy rescaling: the reference max only moves when it must
      const bool grow = mb > m_run + 8.0f;
      const float m_new = grow ? mb : m_run;
      const float alpha = (grow && m_run != NEG_INF) ? exp2f(m_run - m_new) : 1.0f;
      const float m_use = m_new == NEG_INF ? 0.f : m_new;
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        s[c] = exp2f(s[c] - m_use);
        ls += s[c];
      }
      l_run = l_run * alpha + ls;
      m_run = m_new;
      // P V of the previous block must be done: it reads the P buffer and
      // accumulates into the O that may need rescaling
      if (i > 0) {
        if (!warp_wait(o_done, (i - 1) & 1, p.err, ERR_A_SOFT, abort)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
          for (int c0 = 0; c0 < nO; c0 += 32) {
            float v[32];
            tc::tmem_ld32(tO + c0 + lane_off, v);
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] *= alpha;
            tmem_st32(tO + c0 + lane_off, v);
          }
        }
      }
      store_row_sw128(sbase + SM::P_OFF, row, s);
      fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(p_full);
    }
    // ---------------- epilogue ----------------
    if (ok && warp_wait(o_done, (nb - 1) & 1, p.err, ERR_A_SOFT, abort)) {
      tc::tc_fence_after();
      const int grow_ = r0 + row;
      const float il = 1.0f / l_run;
      for (int c0 = 0; c0 < nO; c0 += 32) {
        float v[32];
        tc::tmem_ld32(tO + c0 + lane_off, v);
        if (grow_ < p.n) {
          bf16* dst = p.o + (int64_t)grow_ * p.ldo + (int64_t)h * p.hd + c0;
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            if (c0 + k < p.hd) {
              uint4 u;
              u.x = pack_bf16(v[k] * il, v[k + 1] * il);
              u.y = pack_bf16(v[k + 2] * il, v[k + 3] * il);
              u.z = pack_bf16(v[k + 4] * il, v[k + 5] * il);
              u.w = pack_bf16(v[k + 6] * il, v[k + 7] * il);
              *reinterpret_cast<uint4*>(dst + k) = u;
            }
          }
        }
      }
      if (grow_ < p.n) p.lse[(int64_t)h * p.ld_lse + grow_] = (m_run + log2f(l_run)) * 0.69314718055994531f;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------------------
// Forward for long spans: two query tiles per CTA, P kept in TMEM.
//
// One CTA (1 per SM, all 512 TMEM columns) takes 256 query rows of one head
// as two 128-row tiles t = 0, 1 and walks 128-key blocks:
//   S_t = Q_t K_j^T             (tcgen05, A and B in shared memory)
//   P_t = exp(S_t - m)          (softmax warpgroup t; P written back to
//                                TMEM over the first 64 columns of S_t, two
//                                bf16 per 32-bit column)
//   O_t += P_t V_j              (tcgen05 with A read from TMEM)
// The MMA warp alternates the tiles (after P_0 V_j it issues S_0 of the next
// block, then waits for P_1, ...) so the tensor core computes one tile's
// products while the other tile's softmax runs, and P never passes through
// shared memory.  Because MMAs of one thread complete in issue order, the
// completion of S_t(j) also means P_t(j-1) V has completed: the softmax may
// then overwrite P_t and rescale O_t without further waiting.
// Ten warps: warp 0 loads (TMA), warp 1 issues the MMAs, warps 2-5 and 6-9
// are the softmax warpgroups of tiles 0 and 1, one thread per query row.
// ---------------------------------------------------------------------------
constexpr int BN2 = 128;  // keys per block

template <int NA>
struct Fwd2Smem {
  static constexpr int Q_BYTES = NA * BM * 128;    // one 128-row tile
  static constexpr int KV_BYTES = NA * BN2 * 128;  // one 128-key block
  static constexpr int Q_OFF = 0;                  // two tiles
  static constexpr int K_OFF = 2 * Q_BYTES;
  static constexpr int V_OFF = K_OFF + STAGES * KV_BYTES;
  static constexpr int BAR_OFF = V_OFF + STAGES * KV_BYTES;
  static constexpr int END = BAR_OFF + 256;
  // at least 120 KB: one CTA (512 TMEM columns) per SM
  static constexpr int SMEM = END > 120 * 1024 ? END : 120 * 1024;
};

// 32 lanes x 32 columns, no wait (the caller waits once for several loads)
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 2^x for x <= 0 (the softmax exponent after the row maximum is subtracted):
// the MUFU instruction, subnormal results flushed to zero
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// (a0, a1) * b + c for two lanes of fp32 in one packed instruction
__device__ __forceinline__ void fma2(float a0, float a1, float b, float c, float& d0, float& d1) {
  asm("{\n.reg .b64 ra, rb, rc, rd;\n"
      "mov.b64 ra, {%2, %3};\n"
      "mov.b64 rb, {%4, %4};\n"
      "mov.b64 rc, {%5, %5};\n"
      "fma.rn.f32x2 rd, ra, rb, rc;\n"
      "mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// (a0, a1) * (b0, b1)
__device__ __forceinline__ void mul2(float a0, float a1, float b0, float b1, float& d0, float& d1) {
  asm("{\n.reg .b64 ra, rb, rd;\n"
      "mov.b64 ra, {%2, %3};\n"
      "mov.b64 rb, {%4, %5};\n"
      "mul.rn.f32x2 rd, ra, rb;\n"
      "mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// 32 lanes x 16 columns store (no wait)
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// key-block range of query tile t of the pair starting at row r0 (nb = 0:
// the tile has no rows)
__device__ __forceinline__ void tile2_range(const FwdParams& p, int r0, int t, long long* kb_lo, long long* kb_hi) {
  const int rs = r0 + BM * t;
  if (rs >= p.n) {
    *kb_lo = 1;
    *kb_hi = 0;
    return;
  }
  const long long t_lo = p.pos0 + rs;
  const long long t_hi = p.pos0 + min(rs + BM, p.n) - 1;
  long long k_lo = t_lo - p.W + 1;
  if (k_lo < 0) k_lo = 0;
  *kb_lo = k_lo / BN2;
  *kb_hi = t_hi / BN2;
}

template <int NA>
__global__ void __launch_bounds__(320, 1)
    attn_fwd2_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                        const __grid_constant__ CUtensorMap mapV, FwdParams p) {
  using SM = Fwd2Smem<NA>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + SM::BAR_OFF;
  const uint32_t q_full = bar0;
  const uint32_t k_full = bar0 + 8;     // [2] stages
  const uint32_t v_full = bar0 + 24;    // [2]
  const uint32_t k_empty = bar0 + 40;   // [2] stages: K of the stage consumed
  const uint32_t v_empty = bar0 + 200;  // [2] stages: V of the stage consumed
  const uint32_t s_full = bar0 + 56;    // [2] tiles
  const uint32_t p_full = bar0 + 72;    // [2] tiles
  const uint32_t o_done = bar0 + 88;    // [2] tiles
  const uint32_t drain = bar0 + 104;
  uint32_t* tmem_slot = (uint32_t*)(smem + SM::BAR_OFF + 192);
  volatile int* abort = (volatile int*)(smem + SM::BAR_OFF + 196);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * 2 * BM, h = blockIdx.y, zpart = blockIdx.z;
  const int kvh = h / (p.H / p.Hkv);
  long long lo_t[2], hi_t[2];
  tile2_range(p, r0, 0, &lo_t[0], &hi_t[0]);
  tile2_range(p, r0, 1, &lo_t[1], &hi_t[1]);
  // the pair's key blocks, and this part's share of them
  const long long u_lo = lo_t[0];
  const long long u_hi = hi_t[1] >= lo_t[1] ? max(hi_t[0], hi_t[1]) : hi_t[0];
  const long long nb_all = u_hi - u_lo + 1;
  const long long kb_lo = u_lo + zpart * nb_all / p.parts;
  const int nbl = (int)(u_lo + (zpart + 1) * nb_all / p.parts - kb_lo);
  auto part = [&](int t, long long j) { return j >= lo_t[t] && j <= hi_t[t]; };
  const int ksteps = p.hd / 16;
  const int nO = (p.hd + 15) & ~15;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(k_full + 8 * s, 1);
      tc::mbar_init(v_full + 8 * s, 1);
      tc::mbar_init(k_empty + 8 * s, 1);
      tc::mbar_init(v_empty + 8 * s, 1);
      tc::mbar_init(s_full + 8 * s, 1);
      tc::mbar_init(p_full + 8 * s, 4);  // one arrival per softmax warp of the tile
      tc::mbar_init(o_done + 8 * s, 1);
    }
    tc::mbar_init(drain, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&mapQ);
    tc::prefetch_tmap(&mapK);
    tc::prefetch_tmap(&mapV);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything below reads what earlier kernels wrote
  pdl_wait();
  pdl_trigger();
  // columns: S/P of tile 0 | S/P of tile 1 | O of tile 0 | O of tile 1

  if (warp == 0) {
    if (lane == 0 && nbl > 0) {
      bool ok = true;
      int issued = 0;
      tc::mbar_arrive_expect_tx(q_full, 2 * SM::Q_BYTES);
      for (int t = 0; t < 2; ++t)
        for (int a = 0; a < NA; ++a)
          tma_load_box(KB_ATTN_FWD2_TC, sbase + SM::Q_OFF + t * SM::Q_BYTES + a * BM * 128, &mapQ,
                       h * p.hd + 64 * a, r0 + BM * t, p.H * p.hd, p.n, BM, 0, q_full, abort);
      for (int i = 0; i < nbl && ok; ++i) {
        const int st = i & 1;
        // K and V of a stage are released separately: K once both tiles'
        // scores of its block are done, V once both P.V products are, so
        // the next K lands a block earlier than with one shared release
        if (!tc::mbar_wait(k_empty + 8 * st, ((i >> 1) & 1) ^ 1, p.err, ERR_A_PROD, abort)) {
          ok = false;
          break;
        }
        const long long kpos = (kb_lo + i) * BN2;
        const int row = kvh * p.R + (int)(kpos % p.R);
        tc::mbar_arrive_expect_tx(k_full + 8 * st, SM::KV_BYTES);
        for (int a = 0; a < NA; ++a)
          tma_load_box(KB_ATTN_FWD2_TC, sbase + SM::K_OFF + st * SM::KV_BYTES + a * BN2 * 128, &mapK, 64 * a, row,
                       p.hd, p.Hkv * p.R, BN2, p.R, k_full + 8 * st, abort);
        if (!tc::mbar_wait(v_empty + 8 * st, ((i >> 1) & 1) ^ 1, p.err, ERR_A_PROD, abort)) {
          ok = false;
          break;
        }
        tc::mbar_arrive_expect_tx(v_full + 8 * st, SM::KV_BYTES);
        for (int a = 0; a < NA; ++a)
          tma_load_box(KB_ATTN_FWD2_TC, sbase + SM::V_OFF + st * SM::KV_BYTES + a * BN2 * 128, &mapV, 64 * a, row,
                       p.hd, p.Hkv * p.R, BN2, p.R, v_full + 8 * st, abort);
        issued = i + 1;
      }
      const long long t0 = clock64();
      while (!tc::mbar_try_wait(q_full, 0) && clock64() - t0 < tc::kWaitClocks) {
      }
      for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i) {
        const int st = i & 1;
        const uint32_t par = (i >> 1) & 1;
        const long long t1 = clock64();
        while (!(tc::mbar_try_wait(k_full + 8 * st, par) && tc::mbar_try_wait(v_full + 8 * st, par)) &&
               clock64() - t1 < tc::kWaitClocks) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nbl > 0) {
      const uint32_t idS = tc::idesc_bf16(BM, BN2, 0, 0);
      const uint32_t idO = tc::idesc_bf16(BM, nO, 0, 1);
      bool ok = tc::mbar_wait(q_full, 0, p.err, ERR_A_MMA, abort);
      bool issued = false;
      int cnt[2] = {0, 0};
      // S_t of block i (K of stage i & 1 must have landed)
      auto issue_s = [&](int t, int i) -> bool {
        const int st = i & 1;
        if (!tc::mbar_wait(k_full + 8 * st, (i >> 1) & 1, p.err, ERR_A_MMA, abort)) return false;
        tc::tc_fence_after();
        const uint32_t kb = sbase + SM::K_OFF + st * SM::KV_BYTES;
        const uint32_t qb = sbase + SM::Q_OFF + t * SM::Q_BYTES;
        for (int j = 0; j < ksteps; ++j) {
          const int a = j >> 2;
          tc::mma_bf16(tmem + 128 * t, tc::smem_desc_sw128(qb + a * BM * 128 + 32 * (j & 3), 16, 1024),
                       tc::smem_desc_sw128(kb + a * BN2 * 128 + 32 * (j & 3), 16, 1024), idS, j > 0);
        }
        tc::mma_commit(s_full + 8 * t);
        issued = true;
        return true;
      };
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (ok && nbl > 0 && part(t, kb_lo)) ok = issue_s(t, 0);
      if (ok && nbl > 0) tc::mma_commit(k_empty);
      for (int i = 0; i < nbl && ok; ++i) {
        const long long j = kb_lo + i;
        const int st = i & 1;
        if (!tc::mbar_wait(v_full + 8 * st, (i >> 1) & 1, p.err, ERR_A_MMA, abort)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok) break;
          if (part(t, j)) {
            if (!tc::mbar_wait(p_full + 8 * t, cnt[t] & 1, p.err, ERR_A_MMA, abort)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
            const uint32_t vb = sbase + SM::V_OFF + st * SM::KV_BYTES;
#pragma unroll
            for (int k = 0; k < BN2 / 16; ++k)
              mma_bf16_ts(tmem + 256 + 128 * t, tmem + 128 * t + 8 * k,
                          tc::smem_desc_sw128(vb + 2048 * k, BN2 * 128, 1024), idO, (cnt[t] > 0 || k > 0) ? 1u : 0u);
            tc::mma_commit(o_done + 8 * t);
            ++cnt[t];
          }
          if (t == 1 && ok) tc::mma_commit(v_empty + 8 * st);
          if (ok && i + 1 < nbl && part(t, j + 1)) ok = issue_s(t, i + 1);
        }
        if (ok && i + 1 < nbl) tc::mma_commit(k_empty + 8 * ((i + 1) & 1));
      }
      if (!ok && issued) {
        tc::mma_commit(drain);
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(drain, 0) && clock64() - t0 < tc::kWaitClocks) {
        }
      }
    }
  } else {
    // ---------------- softmax: warps 2-5 tile 0, warps 6-9 tile 1 --------
    // One warp per TMEM lane quarter of a tile, one thread per query row
    // holding all 128 scores of the block in registers: the row maximum
    // needs no exchange between warps, and a warp overwrites only its own
    // rows' scores with their packed P (keys 2c, 2c+1 -> column c).
    const int t = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int grow_ = r0 + BM * t + row;
    const long long pos = p.pos0 + grow_;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + 128 * t + lane_off;
    const uint32_t tO = tmem + 256 + 128 * t + lane_off;
    const float NEG_INF = -INFINITY;
    float m_run = NEG_INF, l_run = 0.f;
    bool ok = true;
    int cnt = 0;
    long long my_lo, my_hi;
    tile2_range(p, r0, t, &my_lo, &my_hi);
    my_lo = max(my_lo, kb_lo);
    my_hi = min(my_hi, kb_lo + nbl - 1);
    for (long long j = my_lo; j <= my_hi; ++j, ++cnt) {
      if (!warp_wait(s_full + 8 * t, cnt & 1, p.err, ERR_A_SOFT, abort)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      float sv[128];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32_nw(tS + 32 * q, *reinterpret_cast<float(*)[32]>(&sv[32 * q]));
      tmem_wait_ld();
      const long long kpos = j * BN2;
      const long long lo_l = pos - p.W + 1 - kpos, hi_l = pos - kpos;
      const int lo = (int)(lo_l < -1 ? -1 : (lo_l > 128 ? 128 : lo_l));
      const int hi = (int)(hi_l < -1 ? -1 : (hi_l > 128 ? 128 : hi_l));
      // maximum of the raw scores (the scale is positive); masked -> -inf
      if (!(lo <= 0 && hi >= 127)) {
#pragma unroll
        for (int c = 0; c < 128; ++c) sv[c] = (c >= lo && c <= hi) ? sv[c] : NEG_INF;
      }
      float mb = NEG_INF;
#pragma unroll
      for (int c = 0; c < 128; c += 2) mb = max3f(mb, sv[c], sv[c + 1]);
      mb *= p.scale_log2;
      const bool grow = mb > m_run + 8.0f;
      const float m_new = grow ? mb : m_run;
      const float alpha = (grow && m_run != NEG_INF) ? exp2f(m_run - m_new) : 1.0f;
      const float m_use = m_new == NEG_INF ? 0.f : m_new;
      // P_t(j-1) V has completed (it was issued before S_t(j)): O_t is
      // stable and P_t may be overwritten.
      // p = 2^(s * scale - m): one packed FMA per two scores, one MUFU each
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float x0, x1;
          fma2(sv[32 * q + 2 * c], sv[32 * q + 2 * c + 1], p.scale_log2, -m_use, x0, x1);
          const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
          ls0 += p0;
          ls1 += p1;
          pk[c] = pack_bf16(p0, p1);
        }
        tmem_st16u(tS + 16 * q, pk);
      }
      const float ls = ls0 + ls1;
      l_run = l_run * alpha + ls;
      m_run = m_new;
      if (cnt > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        for (int c0 = 0; c0 < nO; c0 += 32) {
          float v[32];
          tc::tmem_ld32(tO + c0, v);
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] *= alpha;
          tmem_st32(tO + c0, v);
        }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc::tc_fence_before();
      warp_arrive(p_full + 8 * t);
    }
    const float l_tot = l_run;
    if (ok && p.parts > 1) {
      // this part's share: the unnormalised output (zero if the tile saw no
      // key block here) and (max, sum) of the row, merged by the combine
      // kernel
      const bool have = cnt > 0 && warp_wait(o_done + 8 * t, (cnt - 1) & 1, p.err, ERR_A_SOFT, abort);
      if (cnt > 0 && !have) ok = false;
      if (ok) {
        tc::tc_fence_after();
        const int64_t ldw = (int64_t)p.H * p.hd;
        for (int c0 = 0; c0 < nO; c0 += 32) {
          float v[32];
          if (have) {
            tc::tmem_ld32(tO + c0, v);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = 0.f;
          }
          if (grow_ < p.n) {
            float* dst = p.ws + ((int64_t)zpart * p.n + grow_) * ldw + (int64_t)h * p.hd + c0;
#pragma unroll
            for (int k = 0; k < 32; k += 4)
              if (c0 + k < p.hd) *reinterpret_cast<float4*>(dst + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
          }
        }
        if (grow_ < p.n)
          *reinterpret_cast<float2*>(p.ws_ml + (((int64_t)zpart * p.H + h) * p.n + grow_) * 2) =
              make_float2(have ? m_run : NEG_INF, have ? l_tot : 0.f);
      }
    } else if (ok && cnt > 0 && warp_wait(o_done + 8 * t, (cnt - 1) & 1, p.err, ERR_A_SOFT, abort)) {
      tc::tc_fence_after();
      const float il = 1.0f / l_tot;
      for (int c0 = 0; c0 < nO; c0 += 32) {
        float v[32];
        tc::tmem_ld32(tO + c0, v);
        if (grow_ < p.n) {
          bf16* dst = p.o + (int64_t)grow_ * p.ldo + (int64_t)h * p.hd + c0;
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            if (c0 + k < p.hd) {
              uint4 u;
              u.x = pack_bf16(v[k] * il, v[k + 1] * il);
              u.y = pack_bf16(v[k + 2] * il, v[k + 3] * il);
              u.z = pack_bf16(v[k + 4] * il, v[k + 5] * il);
              u.w = pack_bf16(v[k + 6] * il, v[k + 7] * il);
              *reinterpret_cast<uint4*>(dst + k) = u;
            }
          }
        }
      }
      if (grow_ < p.n)
        p.lse[(int64_t)h * p.ld_lse + grow_] = (m_run + log2f(l_tot)) * 0.69314718055994531f;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// backward
//
//   D[t]   = sum_d dO[t,d] O[t,d]                          (attn_bwd_prep)
//   P      = exp(q.k / sqrt(hd) - lse[t])   (masked to the band)
//   dS     = P (dO.v - D[t]) / sqrt(hd)
//   dq[t]  = sum_j dS[t,j] k_j        over the whole window  (dq kernel)
//   dk[j]  = sum_t dS[t,j] q_t,  dv[j] = sum_t P[t,j] dO_t
//            for the chunk's own keys only                   (dkv kernel)
// The dq kernel may split a tile's key range into `parts` (more CTAs than
// SMs for short chunks); partial sums go to fp32 scratch and a reduction
// adds them in a fixed order, so results are deterministic.  The dkv kernel
// works per query head; a second reduction sums the heads of each KV group.
// ---------------------------------------------------------------------------
struct BwdParams {
  int n, H, Hkv, hd, W, R;
  long long pos0;
  float scale_log2;  // log2(e) / sqrt(hd)
  float scale;       // 1 / sqrt(hd)
  const float* lse;  // [H][ld_lse]
  const float* dsum; // [H][ld_lse]
  int ld_lse;
  int parts;         // dq: key-range parts
  bf16* dqkv;
  int64_t ldg;
  float* ws;
  int* err;
  const float2* cs;  // RoPE table [n][hd/2] to rotate dq, dk back with, or null
};

// The transpose of the forward's RoPE rotation on one adjacent column pair
// (the pair-interleaved layout of q and k): (x, y) -> (x c + y s, y c - x s).
__device__ __forceinline__ void rope_back(float& x, float& y, float2 cs) {
  const float x0 = x;
  x = x0 * cs.x + y * cs.y;
  y = y * cs.x - x0 * cs.y;
}


// --- dq: one 128-row query tile per CTA over 128-key blocks ----------------
// A CTA takes 128 query rows of one head (all or a part of their key range)
// over blocks of DQ_BN = 128 keys, so every score product is a
// 128 x 128 x 16 MMA (64-key blocks made them 128 x 64, which the tensor
// core runs at two thirds of its rate).  TMEM: S of block i in buffer
// i & 1 (columns [0, 128) or [384, 512)), dP in [128, 256), dQ in
// [256, 384).  The compute warps turn S and dP into
// dS = P (dP - D) / sqrt(hd), written back as bf16 pairs over score columns
// each warp has read itself (keys 32 ks.. -> columns 32 ks.., 16 wide), and
// the dQ product reads dS from TMEM as its A operand (K = 16 slices at
// columns 32 (k >> 1) + 8 (k & 1)).
// MMA order for block i: S(i + 1) into the other S buffer, dP(i + 1) once
// the compute warps have loaded dP(i) into registers, then dQ(i) once dS(i)
// is ready; so the tensor core computes the next block's scores and dP
// while dS(i) is formed, and dQ(i) while the warps start on block i + 1.
// dS(i) completions alternate between two barriers by block parity, so a
// waiter never sees a phase of the block after next.  Products of one thread run in issue order,
// which keeps every buffer's reader ahead of its next writer.
// Eighteen warps: warp 0 loads (TMA), warp 1 issues the MMAs, warps 2-17
// compute dS (four per TMEM lane quarter, 32 of a block's 128 keys each).
// Keys move through a ring of 3 blocks, values through a ring of 2: a key
// block is released once its dQ product is done, a value block once its dP
// product is.
constexpr int DQ_BN = 128;
constexpr int DQ_KST = 3, DQ_VST = 2;
template <int NA>
struct DqSmem {
  static constexpr int Q_BYTES = NA * BM * 128;      // one 128-row tile
  static constexpr int KV_BYTES = NA * DQ_BN * 128;  // one 128-key block
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = Q_BYTES;
  static constexpr int K_OFF = 2 * Q_BYTES;
  static constexpr int V_OFF = K_OFF + DQ_KST * KV_BYTES;
  static constexpr int BAR_OFF = V_OFF + DQ_VST * KV_BYTES;
  // at least 120 KB: one CTA (512 TMEM columns) per SM
  static constexpr int SMEM = BAR_OFF + 256 > 120 * 1024 ? BAR_OFF + 256 : 120 * 1024;
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(8 + 16 * (DQ_KST + DQ_VST) + 48 <= 192, "barrier area");
};

// key-block range [lo, hi] (blocks of DQ_BN) of the tile starting at row r0
__device__ __forceinline__ void dq_range(const BwdParams& p, int r0, long long* lo, long long* hi) {
  const long long t_lo = p.pos0 + r0;
  const long long t_hi = p.pos0 + min(r0 + BM, p.n) - 1;
  long long k_lo = t_lo - p.W + 1;
  if (k_lo < 0) k_lo = 0;
  *lo = k_lo / DQ_BN;
  *hi = t_hi / DQ_BN;
}

template <int NA>
__global__ void __launch_bounds__(576, 1)
    attn_dq_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapDO,
                      const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                      BwdParams p) {
  using SM = DqSmem<NA>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + SM::BAR_OFF;
  const uint32_t q_full = bar0;
  const uint32_t k_full = bar0 + 8;                // [DQ_KST]
  const uint32_t k_empty = k_full + 8 * DQ_KST;    // [DQ_KST]
  const uint32_t v_full = k_empty + 8 * DQ_KST;    // [DQ_VST]
  const uint32_t v_empty = v_full + 8 * DQ_VST;    // [DQ_VST]
  const uint32_t sdp_full = v_empty + 8 * DQ_VST;  // S(i) and dP(i) done
  const uint32_t ds_full = sdp_full + 8;           // [2]: dS(i) written (block parity)
  const uint32_t dq_done = ds_full + 16;
  const uint32_t drain = dq_done + 8;
  const uint32_t dp_free = drain + 8;              // dP(i) read into registers
  uint32_t* tmem_slot = (uint32_t*)(smem + SM::BAR_OFF + 192);
  volatile int* abort = (volatile int*)(smem + SM::BAR_OFF + 196);
  // ring slot and phase parity of block i in a ring of `st` slots
  auto slot = [](int i, int st) { return i % st; };
  auto par = [](int i, int st) { return (uint32_t)((i / st) & 1); };
  // TMEM column of the S buffer of block i
  auto s_col = [](int i) { return (uint32_t)((i & 1) ? 384 : 0); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * BM, h = blockIdx.y, part = blockIdx.z;
  const int kvh = h / (p.H / p.Hkv);
  long long t_lo_b, t_hi_b;
  dq_range(p, r0, &t_lo_b, &t_hi_b);
  const long long nb_all = t_hi_b - t_lo_b + 1;
  const long long jb = t_lo_b + part * nb_all / p.parts;  // this part's blocks
  const int nb = (int)(t_lo_b + (part + 1) * nb_all / p.parts - jb);
  const int ksteps = p.hd / 16;
  const int nO = (p.hd + 15) & ~15;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < DQ_KST; ++s) {
      tc::mbar_init(k_full + 8 * s, 1);
      tc::mbar_init(k_empty + 8 * s, 1);
    }
    for (int s = 0; s < DQ_VST; ++s) {
      tc::mbar_init(v_full + 8 * s, 1);
      tc::mbar_init(v_empty + 8 * s, 1);
    }
    tc::mbar_init(sdp_full, 1);
    tc::mbar_init(ds_full, 16);  // one arrival per compute warp
    tc::mbar_init(ds_full + 8, 16);
    tc::mbar_init(dq_done, 1);
    tc::mbar_init(drain, 1);
    tc::mbar_init(dp_free, 16);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&mapQ);
    tc::prefetch_tmap(&mapDO);
    tc::prefetch_tmap(&mapK);
    tc::prefetch_tmap(&mapV);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything below reads what earlier kernels wrote
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0 && nb > 0) {
      bool ok = true;
      int issued_k = 0, issued_v = 0;
      tc::mbar_arrive_expect_tx(q_full, 2 * SM::Q_BYTES);
      for (int a = 0; a < NA; ++a) {
        tma_load_box(KB_ATTN_DQ_TC, sbase + SM::Q_OFF + a * BM * 128, &mapQ, h * p.hd + 64 * a, r0,
                     p.H * p.hd, p.n, BM, 0, q_full, abort);
        tma_load_box(KB_ATTN_DQ_TC, sbase + SM::DO_OFF + a * BM * 128, &mapDO, h * p.hd + 64 * a, r0,
                     p.H * p.hd, p.n, BM, 0, q_full, abort);
      }
      for (int i = 0; i < nb && ok; ++i) {
        const long long kpos = (jb + i) * DQ_BN;
        const int row = kvh * p.R + (int)(kpos % p.R);
        const int ks = slot(i, DQ_KST), vs = slot(i, DQ_VST);
        if (!tc::mbar_wait(k_empty + 8 * ks, par(i, DQ_KST) ^ 1, p.err, ERR_A_PROD, abort)) {
          ok = false;
          break;
        }
        tc::mbar_arrive_expect_tx(k_full + 8 * ks, SM::KV_BYTES);
        for (int a = 0; a < NA; ++a)
          tma_load_box(KB_ATTN_DQ_TC, sbase + SM::K_OFF + ks * SM::KV_BYTES + a * DQ_BN * 128, &mapK, 64 * a, row,
                       p.hd, p.Hkv * p.R, DQ_BN, p.R, k_full + 8 * ks, abort);
        issued_k = i + 1;
        if (!tc::mbar_wait(v_empty + 8 * vs, par(i, DQ_VST) ^ 1, p.err, ERR_A_PROD, abort)) {
          ok = false;
          break;
        }
        tc::mbar_arrive_expect_tx(v_full + 8 * vs, SM::KV_BYTES);
        for (int a = 0; a < NA; ++a)
          tma_load_box(KB_ATTN_DQ_TC, sbase + SM::V_OFF + vs * SM::KV_BYTES + a * DQ_BN * 128, &mapV, 64 * a, row,
                       p.hd, p.Hkv * p.R, DQ_BN, p.R, v_full + 8 * vs, abort);
        issued_v = i + 1;
      }
      // the CTA must not exit with copies into its shared memory in flight
      // (bounded: a failed role has already set the error word)
      const long long t0 = clock64();
      while (!tc::mbar_try_wait(q_full, 0) && clock64() - t0 < tc::kWaitClocks) {
      }
      for (int i = (issued_k > DQ_KST ? issued_k - DQ_KST : 0); i < issued_k; ++i) {
        const long long t1 = clock64();
        while (!tc::mbar_try_wait(k_full + 8 * slot(i, DQ_KST), par(i, DQ_KST)) &&
               clock64() - t1 < tc::kWaitClocks) {
        }
      }
      for (int i = (issued_v > DQ_VST ? issued_v - DQ_VST : 0); i < issued_v; ++i) {
        const long long t1 = clock64();
        while (!tc::mbar_try_wait(v_full + 8 * slot(i, DQ_VST), par(i, DQ_VST)) &&
               clock64() - t1 < tc::kWaitClocks) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nb > 0) {
      const uint32_t idS = tc::idesc_bf16(BM, DQ_BN, 0, 0);
      const uint32_t idQ = tc::idesc_bf16(BM, nO, 0, 1);
      bool ok = tc::mbar_wait(q_full, 0, p.err, ERR_A_MMA, abort);
      bool issued = false;
      // S(i) = Q K(i)^T into its S buffer
      auto issue_s = [&](int i) -> bool {
        const int ks = slot(i, DQ_KST);
        if (!tc::mbar_wait(k_full + 8 * ks, par(i, DQ_KST), p.err, ERR_A_MMA, abort)) return false;
        tc::tc_fence_after();
        const uint32_t kb = sbase + SM::K_OFF + ks * SM::KV_BYTES;
        for (int j = 0; j < ksteps; ++j) {
          const int a = j >> 2;
          tc::mma_bf16(tmem + s_col(i), tc::smem_desc_sw128(sbase + SM::Q_OFF + a * BM * 128 + 32 * (j & 3), 16, 1024),
                       tc::smem_desc_sw128(kb + a * DQ_BN * 128 + 32 * (j & 3), 16, 1024), idS, j > 0);
        }
        issued = true;
        return true;
      };
      // dP(i) = dO V(i)^T; then S(i) and dP(i) are both on their way to the
      // compute warps, and V(i) is free once dP(i) is done
      auto issue_dp = [&](int i) -> bool {
        const int vs = slot(i, DQ_VST);
        if (!tc::mbar_wait(v_full + 8 * vs, par(i, DQ_VST), p.err, ERR_A_MMA, abort)) return false;
        tc::tc_fence_after();
        const uint32_t vb = sbase + SM::V_OFF + vs * SM::KV_BYTES;
        for (int j = 0; j < ksteps; ++j) {
          const int a = j >> 2;
          tc::mma_bf16(tmem + 128, tc::smem_desc_sw128(sbase + SM::DO_OFF + a * BM * 128 + 32 * (j & 3), 16, 1024),
                       tc::smem_desc_sw128(vb + a * DQ_BN * 128 + 32 * (j & 3), 16, 1024), idS, j > 0);
        }
        tc::mma_commit(sdp_full);
        tc::mma_commit(v_empty + 8 * vs);
        issued = true;
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok) ok = issue_dp(0);
      for (int i = 0; i < nb && ok; ++i) {
        if (i + 1 < nb && !issue_s(i + 1)) {
          ok = false;
          break;
        }
        // dP(i + 1) as soon as the compute warps hold dP(i) in registers,
        // so that it runs while they form dS(i)
        if (i + 1 < nb) {
          if (!tc::mbar_wait(dp_free, (uint32_t)(i & 1), p.err, ERR_A_MMA, abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          if (!issue_dp(i + 1)) {
            ok = false;
            break;
          }
        }
        if (!tc::mbar_wait(ds_full + 8 * (i & 1), (uint32_t)((i >> 1) & 1), p.err, ERR_A_MMA, abort)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const int ks = slot(i, DQ_KST);
        const uint32_t kb = sbase + SM::K_OFF + ks * SM::KV_BYTES;
#pragma unroll
        for (int k = 0; k < DQ_BN / 16; ++k)
          mma_bf16_ts(tmem + 256, tmem + s_col(i) + 32 * (k >> 1) + 8 * (k & 1),
                      tc::smem_desc_sw128(kb + 2048 * k, DQ_BN * 128, 1024), idQ, (i > 0 || k > 0) ? 1u : 0u);
        // K(i) has served S(i) and dQ(i)
        tc::mma_commit(k_empty + 8 * ks);
      }
      if (ok) tc::mma_commit(dq_done);
      if (!ok && issued) {
        tc::mma_commit(drain);
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(drain, 0) && clock64() - t0 < tc::kWaitClocks) {
        }
      }
    }
  } else {
    const int ks = (warp - 2) >> 2;  // key slice [32 ks, 32 ks + 32) of a block
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int grow_ = r0 + row;
    const long long pos = p.pos0 + grow_;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool rvalid = grow_ < p.n;
    const float lse2 = rvalid ? p.lse[(int64_t)h * p.ld_lse + grow_] * 1.4426950408889634f : 0.f;
    const float Dt = rvalid ? p.dsum[(int64_t)h * p.ld_lse + grow_] : 0.f;
    // dS = P (dP - D) / sqrt(hd) = P * (dP * scale - D * scale)
    const float nDs = -Dt * p.scale;
    bool ok = true;
    for (int i = 0; i < nb; ++i) {
      if (!warp_wait(sdp_full, (uint32_t)(i & 1), p.err, ERR_A_SOFT, abort)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const uint32_t ts = tmem + s_col(i) + lane_off + 32 * ks;
      float sv[32], dp[32];
      tmem_ld32_nw(ts, sv);
      tmem_ld32_nw(tmem + 128 + lane_off + 32 * ks, dp);
      tmem_wait_ld();
      // the dP buffer may take dP(i + 1) now
      tc::tc_fence_before();
      warp_arrive(dp_free);
      const long long kpos = (jb + i) * DQ_BN + 32 * ks;
      const long long lo_l = pos - p.W + 1 - kpos, hi_l = pos - kpos;
      const int lo = (int)(lo_l < -1 ? -1 : (lo_l > 32 ? 32 : lo_l));
      const int hi = (int)(hi_l < -1 ? -1 : (hi_l > 32 ? 32 : hi_l));
      uint32_t pk[16];
      if (__all_sync(0xffffffffu, lo <= 0 && hi >= 31)) {
        // every key of the slice is inside every row's window: no mask
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float x0, x1, y0, y1, d0, d1;
          fma2(sv[c], sv[c + 1], p.scale_log2, -lse2, x0, x1);
          fma2(dp[c], dp[c + 1], p.scale, nDs, y0, y1);
          mul2(ex2_ftz(x0), ex2_ftz(x1), y0, y1, d0, d1);
          pk[c / 2] = pack_bf16(d0, d1);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float x0, x1, y0, y1, d0, d1;
          fma2(sv[c], sv[c + 1], p.scale_log2, -lse2, x0, x1);
          const float p0 = (c >= lo && c <= hi) ? ex2_ftz(x0) : 0.f;
          const float p1 = (c + 1 >= lo && c + 1 <= hi) ? ex2_ftz(x1) : 0.f;
          fma2(dp[c], dp[c + 1], p.scale, nDs, y0, y1);
          mul2(p0, p1, y0, y1, d0, d1);
          pk[c / 2] = pack_bf16(d0, d1);
        }
      }
      tmem_st16u(ts, pk);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc::tc_fence_before();
      warp_arrive(ds_full + 8 * (i & 1));
    }
    const bool have = nb > 0;
    if (ok && have && !warp_wait(dq_done, 0, p.err, ERR_A_SOFT, abort)) ok = false;
    const int c0 = 32 * ks;  // this warp's 32 columns of dQ
    if (ok && (have || p.parts > 1) && c0 < nO) {
      tc::tc_fence_after();
      float v[32];
      if (have) {
        tc::tmem_ld32(tmem + 256 + lane_off + c0, v);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = 0.f;
      }
      if (rvalid) {
        if (p.parts == 1) {
          if (p.cs) {
            const float2* csr = p.cs + (int64_t)grow_ * (p.hd >> 1) + (c0 >> 1);
#pragma unroll
            for (int k = 0; k < 32; k += 2)
              if (c0 + k < p.hd) rope_back(v[k], v[k + 1], csr[k >> 1]);
          }
          bf16* dst = p.dqkv + (int64_t)grow_ * p.ldg + (int64_t)h * p.hd + c0;
#pragma unroll
          for (int k = 0; k < 32; k += 8)
            if (c0 + k < p.hd) {
              uint4 u;
              u.x = pack_bf16(v[k], v[k + 1]);
              u.y = pack_bf16(v[k + 2], v[k + 3]);
              u.z = pack_bf16(v[k + 4], v[k + 5]);
              u.w = pack_bf16(v[k + 6], v[k + 7]);
              *reinterpret_cast<uint4*>(dst + k) = u;
            }
        } else {
          float* dst = p.ws + ((int64_t)part * p.n + grow_) * ((int64_t)p.H * p.hd) + (int64_t)h * p.hd + c0;
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            if (c0 + k < p.hd) *reinterpret_cast<float4*>(dst + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
        }
      }
    } else if (ok && have && c0 >= nO) {
      tc::tc_fence_after();
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// --- dk / dv of the chunk's own keys, one CTA per (key tile, query head) ---
template <int NA>
struct DkvSmem {
  static constexpr int T_BYTES = NA * BM * 128;  // 128 key rows
  static constexpr int B_BYTES = NA * BN * 128;  // 64 query rows
  static constexpr int P_BYTES = BM * BN * 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + T_BYTES;
  static constexpr int Q_OFF = V_OFF + T_BYTES;
  static constexpr int DO_OFF = Q_OFF + STAGES * B_BYTES;
  static constexpr int PT_OFF = DO_OFF + STAGES * B_BYTES;
  static constexpr int DS_OFF = PT_OFF + 2 * P_BYTES;
  static constexpr int BAR_OFF = DS_OFF + 2 * P_BYTES;
  static constexpr int SMEM = BAR_OFF + 256 > 120 * 1024 ? BAR_OFF + 256 : 120 * 1024;
};

template <int NA>
__global__ void __launch_bounds__(320, 1)
    attn_dkv_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapDO,
                       const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                       BwdParams p) {
  using SM = DkvSmem<NA>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + SM::BAR_OFF;
  const uint32_t kv_full = bar0;
  const uint32_t q_full = bar0 + 8;      // [2]
  const uint32_t q_empty = bar0 + 24;    // [2]
  const uint32_t s_full = bar0 + 40;     // [2]
  const uint32_t s_empty = bar0 + 56;    // [2]
  const uint32_t pd_full = bar0 + 72;    // [2]
  const uint32_t pd_empty = bar0 + 88;   // [2]
  const uint32_t acc_done = bar0 + 104;
  const uint32_t drain = bar0 + 112;
  uint32_t* tmem_slot = (uint32_t*)(smem + SM::BAR_OFF + 192);
  volatile int* abort = (volatile int*)(smem + SM::BAR_OFF + 196);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, kt = blockIdx.y;
  const int j0 = kt * BM;                       // first key row (chunk-local)
  const int kvh = h / (p.H / p.Hkv);
  const int j_last = min(j0 + BM, p.n) - 1;
  const int t_last = min(p.n - 1, j_last + p.W - 1);
  const int qb0 = j0 / BN;
  const int nb = t_last / BN - qb0 + 1;
  const int ksteps = p.hd / 16;
  const int nO = (p.hd + 15) & ~15;

  if (threadIdx.x == 0) {
    tc::mbar_init(kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(q_full + 8 * s, 1);
      tc::mbar_init(q_empty + 8 * s, 1);
      tc::mbar_init(s_full + 8 * s, 1);
      tc::mbar_init(s_empty + 8 * s, 8);  // one arrival per compute warp
      tc::mbar_init(pd_full + 8 * s, 8);
      tc::mbar_init(pd_empty + 8 * s, 1);
    }
    tc::mbar_init(acc_done, 1);
    tc::mbar_init(drain, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&mapQ);
    tc::prefetch_tmap(&mapDO);
    tc::prefetch_tmap(&mapK);
    tc::prefetch_tmap(&mapV);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything below reads what earlier kernels wrote
  pdl_wait();
  pdl_trigger();
  const uint32_t tS = tmem, tP = tmem + 128, tK = tmem + 256, tV = tmem + 384;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      // the tile's keys and values: two 64-row boxes per atom (chunk starts
      // are multiples of 64, so each box is contiguous in the ring)
      tc::mbar_arrive_expect_tx(kv_full, 2 * SM::T_BYTES);
      for (int m = 0; m < 2; ++m) {
        const int row = kvh * p.R + (int)((p.pos0 + j0 + 64 * m) % p.R);
        for (int a = 0; a < NA; ++a) {
          tma_load_box(KB_ATTN_DKV_TC, sbase + SM::K_OFF + a * BM * 128 + m * 64 * 128, &mapK, 64 * a, row,
                       p.hd, p.Hkv * p.R, 64, p.R, kv_full, abort);
          tma_load_box(KB_ATTN_DKV_TC, sbase + SM::V_OFF + a * BM * 128 + m * 64 * 128, &mapV, 64 * a, row,
                       p.hd, p.Hkv * p.R, 64, p.R, kv_full, abort);
        }
      }
      for (int i = 0; i < nb && ok; ++i) {
        const int st = i & 1;
        if (!tc::mbar_wait(q_empty + 8 * st, ((i >> 1) & 1) ^ 1, p.err, ERR_A_PROD, abort)) {
          ok = false;
          break;
        }
        const int t0 = (qb0 + i) * BN;
        tc::mbar_arrive_expect_tx(q_full + 8 * st, 2 * SM::B_BYTES);
        for (int a = 0; a < NA; ++a) {
          tma_load_box(KB_ATTN_DKV_TC, sbase + SM::Q_OFF + st * SM::B_BYTES + a * BN * 128, &mapQ,
                       h * p.hd + 64 * a, t0, p.H * p.hd, p.n, BN, 0, q_full + 8 * st, abort);
          tma_load_box(KB_ATTN_DKV_TC, sbase + SM::DO_OFF + st * SM::B_BYTES + a * BN * 128, &mapDO,
                       h * p.hd + 64 * a, t0, p.H * p.hd, p.n, BN, 0, q_full + 8 * st, abort);
        }
        issued = i + 1;
      }
      const long long t0 = clock64();
      while (!tc::mbar_try_wait(kv_full, 0) && clock64() - t0 < tc::kWaitClocks) {
      }
      for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i) {
        const long long t1 = clock64();
        while (!tc::mbar_try_wait(q_full + 8 * (i & 1), (i >> 1) & 1) && clock64() - t1 < tc::kWaitClocks) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idS = tc::idesc_bf16(BM, BN, 0, 0);
      const uint32_t idA = tc::idesc_bf16(BM, nO, 0, 1);
      bool ok = tc::mbar_wait(kv_full, 0, p.err, ERR_A_MMA, abort);
      bool issued = false;
      for (int i = 0; i <= nb && ok; ++i) {
        if (i < nb) {
          const int st = i & 1;
          const uint32_t par = (i >> 1) & 1;
          if (!tc::mbar_wait(q_full + 8 * st, par, p.err, ERR_A_MMA, abort) ||
              !tc::mbar_wait(s_empty + 8 * st, par ^ 1, p.err, ERR_A_MMA, abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t qb = sbase + SM::Q_OFF + st * SM::B_BYTES;
          const uint32_t ob = sbase + SM::DO_OFF + st * SM::B_BYTES;
          for (int j = 0; j < ksteps; ++j) {
            const int a = j >> 2;
            const uint32_t ao = a * BM * 128 + 32 * (j & 3);
            const uint32_t bo = a * BN * 128 + 32 * (j & 3);
            tc::mma_bf16(tS + st * BN, tc::smem_desc_sw128(sbase + SM::K_OFF + ao, 16, 1024),
                         tc::smem_desc_sw128(qb + bo, 16, 1024), idS, j > 0);
            tc::mma_bf16(tP + st * BN, tc::smem_desc_sw128(sbase + SM::V_OFF + ao, 16, 1024),
                         tc::smem_desc_sw128(ob + bo, 16, 1024), idS, j > 0);
          }
          issued = true;
          tc::mma_commit(s_full + 8 * st);
        }
        if (i >= 1) {
          const int k = i - 1;
          const int st = k & 1;
          if (!tc::mbar_wait(pd_full + 8 * st, (k >> 1) & 1, p.err, ERR_A_MMA, abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t qb = sbase + SM::Q_OFF + st * SM::B_BYTES;
          const uint32_t ob = sbase + SM::DO_OFF + st * SM::B_BYTES;
#pragma unroll
          for (int j = 0; j < BN / 16; ++j) {
            const uint32_t acc = (k > 0 || j > 0) ? 1u : 0u;
            tc::mma_bf16(tV, tc::smem_desc_sw128(sbase + SM::PT_OFF + st * SM::P_BYTES + 32 * j, 16, 1024),
                         tc::smem_desc_sw128(ob + 2048 * j, BN * 128, 1024), idA, acc);
            tc::mma_bf16(tK, tc::smem_desc_sw128(sbase + SM::DS_OFF + st * SM::P_BYTES + 32 * j, 16, 1024),
                         tc::smem_desc_sw128(qb + 2048 * j, BN * 128, 1024), idA, acc);
          }
          tc::mma_commit(pd_empty + 8 * st);
          tc::mma_commit(q_empty + 8 * st);
        }
      }
      if (ok) tc::mma_commit(acc_done);
      if (!ok && issued) {
        tc::mma_commit(drain);
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(drain, 0) && clock64() - t0 < tc::kWaitClocks) {
        }
      }
    }
  } else {
    // eight compute warps: two per TMEM lane quarter, each taking one half
    // (32 query columns) of the block and of dk / dv's head dimension
    const int quarter = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const int j = j0 + row;                  // chunk-local key index
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float* lse_h = p.lse + (int64_t)h * p.ld_lse;
    const float* d_h = p.dsum + (int64_t)h * p.ld_lse;
    bool ok = true;
    for (int i = 0; i < nb; ++i) {
      const int st = i & 1;
      const uint32_t par = (i >> 1) & 1;
      if (!warp_wait(s_full + 8 * st, par, p.err, ERR_A_SOFT, abort)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const int t0 = (qb0 + i) * BN + 32 * hf;
      uint32_t pp[16], pd[16];
      {
        // lane c holds the statistics of query t0 + c; the loop below
        // takes them by shuffle (every lane needs all 32)
        const int tl = t0 + lane;
        const float l2_l = tl < p.n ? lse_h[tl] * 1.4426950408889634f : 0.f;
        const float nDs_l = tl < p.n ? -d_h[tl] * p.scale : 0.f;
        float sv[32], dp[32];
        tmem_ld32_nw(tS + st * BN + 32 * hf + lane_off, sv);
        tmem_ld32_nw(tP + st * BN + 32 * hf + lane_off, dp);
        tmem_wait_ld();
        // every (key, query) pair of the warp's block is valid: no mask
        const bool all_valid = __all_sync(0xffffffffu, t0 + 31 < p.n && j < p.n && t0 - j >= 0 && t0 + 31 - j < p.W);
        if (all_valid) {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float pv[2], dv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float l2 = __shfl_sync(0xffffffffu, l2_l, c + e);
              const float nDs = __shfl_sync(0xffffffffu, nDs_l, c + e);
              pv[e] = ex2_ftz(fmaf(sv[c + e], p.scale_log2, -l2));
              dv[e] = pv[e] * fmaf(dp[c + e], p.scale, nDs);
            }
            pp[c / 2] = pack_bf16(pv[0], pv[1]);
            pd[c / 2] = pack_bf16(dv[0], dv[1]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float pv[2], dv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int t = t0 + c + e;
              const int rel = t - j;
              const bool valid = t < p.n && j < p.n && rel >= 0 && rel < p.W;
              const float l2 = __shfl_sync(0xffffffffu, l2_l, c + e);
              const float nDs = __shfl_sync(0xffffffffu, nDs_l, c + e);
              pv[e] = valid ? ex2_ftz(fmaf(sv[c + e], p.scale_log2, -l2)) : 0.f;
              dv[e] = valid ? pv[e] * fmaf(dp[c + e], p.scale, nDs) : 0.f;
            }
            pp[c / 2] = pack_bf16(pv[0], pv[1]);
            pd[c / 2] = pack_bf16(dv[0], dv[1]);
          }
        }
      }
      tc::tc_fence_before();
      warp_arrive(s_empty + 8 * st);
      if (!warp_wait(pd_empty + 8 * st, par ^ 1, p.err, ERR_A_SOFT, abort)) {
        ok = false;
        break;
      }
      {
        const uint32_t bp = sbase + SM::PT_OFF + st * SM::P_BYTES + row * 128;
        const uint32_t bd = sbase + SM::DS_OFF + st * SM::P_BYTES + row * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t off = ((4 * hf + c) ^ (row & 7)) << 4;
          st_shared_v4(bp + off, pp[4 * c], pp[4 * c + 1], pp[4 * c + 2], pp[4 * c + 3]);
          st_shared_v4(bd + off, pd[4 * c], pd[4 * c + 1], pd[4 * c + 2], pd[4 * c + 3]);
        }
      }
      fence_proxy_async_smem();
      tc::tc_fence_before();
      warp_arrive(pd_full + 8 * st);
    }
    if (ok && warp_wait(acc_done, 0, p.err, ERR_A_SOFT, abort)) {
      tc::tc_fence_after();
      // per-head partials: ws[0][h][j][:] = dk, ws[1][h][j][:] = dv
      const int64_t plane = (int64_t)p.H * p.n * p.hd;
      for (int c0 = 32 * hf; c0 < nO; c0 += 64) {
        float vk[32], vv[32];
        tc::tmem_ld32(tK + c0 + lane_off, vk);
        tc::tmem_ld32(tV + c0 + lane_off, vv);
        if (j < p.n) {
          float* dkp = p.ws + ((int64_t)h * p.n + j) * p.hd + c0;
          float* dvp = dkp + plane;
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            if (c0 + k < p.hd) {
              *reinterpret_cast<float4*>(dkp + k) = make_float4(vk[k], vk[k + 1], vk[k + 2], vk[k + 3]);
              *reinterpret_cast<float4*>(dvp + k) = make_float4(vv[k], vv[k + 1], vv[k + 2], vv[k + 3]);
            }
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// Merge the key-range parts of the split forward, in part order: with
// M = max_z m_z and L = sum_z 2^(m_z - M) l_z,
//   o = sum_z 2^(m_z - M) O_z / L,   lse = (M + log2 L) ln 2.
// One warp per (row, head); each lane takes hd / 32 columns.
__global__ void attn_fwd_combine_kernel(const float* __restrict__ ws, const float* __restrict__ ws_ml, int parts,
                                        int n, int H, int hd, bf16* __restrict__ o, int64_t ldo,
                                        float* __restrict__ lse, int ld_lse) {
  pdl_wait();
  pdl_trigger();
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= n * H) return;
  const int r = w / H, h = w % H;
  auto ml_of = [&](int z) {
    return *reinterpret_cast<const float2*>(ws_ml + (((int64_t)z * H + h) * n + r) * 2);
  };
  float M = -INFINITY;
  for (int z = 0; z < parts; ++z) M = fmaxf(M, ml_of(z).x);
  const float Mu = M == -INFINITY ? 0.f : M;
  float L = 0.f;
  for (int z = 0; z < parts; ++z) {
    const float2 ml = ml_of(z);
    L += (ml.x == -INFINITY ? 0.f : exp2f(ml.x - Mu)) * ml.y;
  }
  const float il = L > 0.f ? 1.0f / L : 0.f;
  const int64_t ldw = (int64_t)H * hd;
  for (int c = 4 * lane; c < hd; c += 128) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    for (int z = 0; z < parts; ++z) {
      const float mz = ml_of(z).x;
      const float sc = mz == -INFINITY ? 0.f : exp2f(mz - Mu);
      const float4 v = *reinterpret_cast<const float4*>(ws + ((int64_t)z * n + r) * ldw + (int64_t)h * hd + c);
      a0 = fmaf(sc, v.x, a0);
      a1 = fmaf(sc, v.y, a1);
      a2 = fmaf(sc, v.z, a2);
      a3 = fmaf(sc, v.w, a3);
    }
    uint2 u;
    u.x = pack_bf16(a0 * il, a1 * il);
    u.y = pack_bf16(a2 * il, a3 * il);
    *reinterpret_cast<uint2*>(o + (int64_t)r * ldo + (int64_t)h * hd + c) = u;
  }
  if (lane == 0) lse[(int64_t)h * ld_lse + r] = (M + log2f(L)) * 0.69314718055994531f;
}

// D[h][r] = sum_d dO[r, h*hd + d] * O[r, h*hd + d]; one warp per (r, h)
__global__ void attn_bwd_prep_tc_kernel(const bf16* __restrict__ dO, const bf16* __restrict__ O, int n, int H,
                                        int hd, float* __restrict__ dsum, int ld) {
  pdl_wait();
  pdl_trigger();
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= n * H) return;
  const int r = w / H, h = w % H;
  const int64_t off = (int64_t)r * H * hd + (int64_t)h * hd;
  float s = 0.f;
  for (int d = 2 * lane; d < hd; d += 64) {
    const float2 a = load2<bf16>(dO + off + d);
    const float2 b = load2<bf16>(O + off + d);
    s = fmaf(a.x, b.x, fmaf(a.y, b.y, s));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) dsum[(int64_t)h * ld + r] = s;
}

// dq = sum over parts (fixed order) -> bf16 columns [0, H*hd) of dqkv,
// rotated back by the RoPE table cs when given
__global__ void attn_dq_reduce_kernel(const float* __restrict__ ws, int parts, int n, int cols,
                                      bf16* __restrict__ dqkv, int64_t ldg, const float2* __restrict__ cs,
                                      int hd) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)n * cols / 4;
  const int64_t plane = (int64_t)n * cols;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = 4 * i;
    float4 acc = *reinterpret_cast<const float4*>(ws + e);
    for (int q = 1; q < parts; ++q) {
      const float4 v = *reinterpret_cast<const float4*>(ws + q * plane + e);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int64_t r = e / cols, c = e % cols;
    if (cs) {
      const float2* csr = cs + r * (hd >> 1) + ((c % hd) >> 1);
      rope_back(acc.x, acc.y, csr[0]);
      rope_back(acc.z, acc.w, csr[1]);
    }
    bf16* d = dqkv + r * ldg + c;
    *reinterpret_cast<uint2*>(d) = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
  }
}

// dk, dv of KV head g = sum over its query heads (fixed order) -> bf16;
// dk rotated back by the RoPE table cs when given
__global__ void attn_dkv_reduce_kernel(const float* __restrict__ ws, int n, int H, int Hkv, int hd,
                                       bf16* __restrict__ dqkv, int64_t ldg, const float2* __restrict__ cs) {
  pdl_wait();
  pdl_trigger();
  const int group = H / Hkv;
  const int64_t total = (int64_t)2 * n * Hkv * hd / 4;
  const int64_t plane = (int64_t)H * n * hd;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    int64_t e = 4 * i;
    const int which = (int)(e / ((int64_t)n * Hkv * hd));   // 0 dk, 1 dv
    e -= (int64_t)which * n * Hkv * hd;
    const int r = (int)(e / ((int64_t)Hkv * hd));
    const int g = (int)((e / hd) % Hkv);
    const int d = (int)(e % hd);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < group; ++k) {
      const int h = g * group + k;
      const float4 v = *reinterpret_cast<const float4*>(ws + which * plane + ((int64_t)h * n + r) * hd + d);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (cs && which == 0) {
      const float2* csr = cs + (int64_t)r * (hd >> 1) + (d >> 1);
      rope_back(acc.x, acc.y, csr[0]);
      rope_back(acc.z, acc.w, csr[1]);
    }
    bf16* dst = dqkv + (int64_t)r * ldg + (int64_t)(H + which * Hkv + g) * hd + d;
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
  }
}

// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;
std::once_flag g_enc_once;

bool encoder() {
  std::call_once(g_enc_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_enc = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  });
  return g_enc != nullptr;
}

// bf16 2-D map: inner extent `inner` (elements, contiguous), `outer` rows of
// pitch `ld` elements, box {64, box_rows}, 128-byte swizzle, zero fill
int map2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

// Key-range parts of a kernel whose CTA takes rows_per_cta query rows of a
// head over blocks of bn keys: enough CTAs to fill the SMs in whole waves,
// never more parts than the smallest tile has key blocks, at most max_parts.
// Each further part costs `overhead` of a CTA's work (its prologue, the
// partial results and their merge).
static int split_parts(const AttnArgs& a, int num_sms, int rows_per_cta, int bn, int max_parts,
                       double overhead) {
  const int ntiles = (a.n + rows_per_cta - 1) / rows_per_cta;
  int nb_min = INT32_MAX;
  for (int t = 0; t < ntiles; ++t) {
    const long long t_lo = a.pos0 + (long long)t * rows_per_cta;
    const long long t_hi = a.pos0 + std::min(t * rows_per_cta + rows_per_cta, a.n) - 1;
    long long k_lo = t_lo - a.W + 1;
    if (k_lo < 0) k_lo = 0;
    nb_min = std::min<int>(nb_min, (int)(t_hi / bn - k_lo / bn + 1));
  }
  const int units = ntiles * a.H;
  int best = 1;
  double best_cost = 1e30;
  for (int P = 1; P <= max_parts && P <= nb_min; ++P) {
    const double waves = std::ceil((double)units * P / num_sms);
    const double cost = waves / P * (1.0 + overhead * (P - 1));
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = P;
    }
  }
  return best;
}

template <int NA>
int launch_fwd(const AttnArgs& a, int* err, cudaStream_t st) {
  using SM = FwdSmem<NA>;
  CUtensorMap mq, mk, mv;
  const uint64_t ldq = (uint64_t)a.H * a.hd;
  int rc = map2d(&mq, a.q, ldq, a.n, ldq, BM);
  if (!rc) rc = map2d(&mk, a.kring, a.hd, (uint64_t)a.Hkv * a.R, a.hd, BN);
  if (!rc) rc = map2d(&mv, a.vring, a.hd, (uint64_t)a.Hkv * a.R, a.hd, BN);
  if (rc) return rc;
  static std::atomic<uint64_t> attr{0};
  {
    cudaError_t e = raise_smem_limit(attr, attn_fwd_tc_kernel<NA>, SM::SMEM);
    if (e != cudaSuccess) return (int)e;
  }
  FwdParams p;
  p.n = a.n;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.hd = a.hd;
  p.W = a.W;
  p.R = a.R;
  p.pos0 = a.pos0;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)a.hd);
  p.o = (bf16*)a.o;
  p.ldo = (int64_t)a.H * a.hd;
  p.lse = a.lse;
  p.ld_lse = a.ld_lse;
  p.err = err;
  p.parts = 1;
  p.ws = p.ws_ml = nullptr;
  dim3 grid((a.n + BM - 1) / BM, a.H);
  launch_k(attn_fwd_tc_kernel<NA>, grid, 192, SM::SMEM, st, mq, mk, mv, p);
  return (int)cudaPeekAtLastError();
}

template <int NA>
int launch_fwd2(const AttnArgs& a, int* err, cudaStream_t st, int* kernels) {
  using SM = Fwd2Smem<NA>;
  CUtensorMap mq, mk, mv;
  const uint64_t ldq = (uint64_t)a.H * a.hd;
  int rc = map2d(&mq, a.q, ldq, a.n, ldq, BM);
  if (!rc) rc = map2d(&mk, a.kring, a.hd, (uint64_t)a.Hkv * a.R, a.hd, BN2);
  if (!rc) rc = map2d(&mv, a.vring, a.hd, (uint64_t)a.Hkv * a.R, a.hd, BN2);
  if (rc) return rc;
  static std::atomic<uint64_t> attr{0};
  {
    cudaError_t e = raise_smem_limit(attr, attn_fwd2_tc_kernel<NA>, SM::SMEM);
    if (e != cudaSuccess) return (int)e;
  }
  FwdParams p;
  p.n = a.n;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.hd = a.hd;
  p.W = a.W;
  p.R = a.R;
  p.pos0 = a.pos0;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)a.hd);
  p.o = (bf16*)a.o;
  p.ldo = (int64_t)a.H * a.hd;
  p.lse = a.lse;
  p.ld_lse = a.ld_lse;
  p.err = err;
  // with scratch, split the key range when the tile pairs alone leave SMs
  // idle (a chunk of 1024 rows has 4 pairs per head)
  p.parts = 1;
  p.ws = p.ws_ml = nullptr;
  if (a.ws) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t plane = (int64_t)a.n * a.H * a.hd, ml = (int64_t)2 * a.n * a.H;
    // measured at the 3B shapes: 3 parts beat 1 at 1024 rows (96 tile pairs
    // for 148 SMs) and lose at 4096 rows, where the pairs fill 2.6 waves
    int parts = split_parts(a, sms, 2 * BM, BN2, 3, 0.08);
    while (parts > 1 && (int64_t)parts * (plane + ml) > a.ws_elems) --parts;
    if (parts > 1) {
      p.parts = parts;
      p.ws = a.ws;
      p.ws_ml = a.ws + (int64_t)parts * plane;
    }
  }
  dim3 grid((a.n + 2 * BM - 1) / (2 * BM), a.H, p.parts);
  launch_k(attn_fwd2_tc_kernel<NA>, grid, 320, SM::SMEM, st, mq, mk, mv, p);
  if (kernels) *kernels = p.parts > 1 ? 2 : 1;
  if (p.parts > 1) {
    const int64_t warps = (int64_t)a.n * a.H;
    launch_k(attn_fwd_combine_kernel, (int)((warps + 7) / 8), 256, 0, st, p.ws, p.ws_ml, p.parts, a.n, a.H, a.hd, p.o,
                                                                      p.ldo, a.lse, a.ld_lse);
  }
  return (int)cudaPeekAtLastError();
}

}  // namespace

bool attn_tc_supported(const AttnArgs& a) {
  return a.hd >= 64 && a.hd <= 128 && a.hd % 16 == 0 && a.R % 128 == 0 && a.H % a.Hkv == 0 &&
         ((uintptr_t)a.q & 15) == 0 && ((uintptr_t)a.kring & 15) == 0 && ((uintptr_t)a.vring & 15) == 0 &&
         ((uintptr_t)a.o & 15) == 0;
}

int attn_fwd_tc(const AttnArgs& a, int* err, cudaStream_t st, int variant, int* kernels) {
  if (kernels) *kernels = 1;
  if (a.n <= 0) return 0;
  if (!encoder() || !attn_tc_supported(a)) return (int)cudaErrorNotSupported;
  // the two-tile kernel measured faster at every size tried (1K and 16K
  // rows, head dims 64 and 128)
  if (variant == 0) variant = 2;
  if (variant == 2) return a.hd <= 64 ? launch_fwd2<1>(a, err, st, kernels) : launch_fwd2<2>(a, err, st, kernels);
  return a.hd <= 64 ? launch_fwd<1>(a, err, st) : launch_fwd<2>(a, err, st);
}

int64_t attn_bwd_tc_ws_elems(int n, int H, int hd, int num_sms) {
  (void)num_sms;
  // up to 4 planes of dq key-range partials, then 2 of dk / dv partials
  // (dk/dv beside dq); 2 planes are the least the kernels need
  return (int64_t)6 * n * H * hd;
}

template <int NA>
int launch_bwd(const AttnArgs& a, int* err, cudaStream_t st, int num_sms) {
  using DQ = DqSmem<NA>;
  using DKV = DkvSmem<NA>;
  CUtensorMap mq, mdo, mk, mv, mq64, mdo64, mk128, mv128;
  const uint64_t ldq = (uint64_t)a.H * a.hd;
  int rc = map2d(&mq, a.q, ldq, a.n, ldq, BM);
  if (!rc) rc = map2d(&mdo, a.dout, ldq, a.n, ldq, BM);
  if (!rc) rc = map2d(&mq64, a.q, ldq, a.n, ldq, BN);
  if (!rc) rc = map2d(&mdo64, a.dout, ldq, a.n, ldq, BN);
  if (!rc) rc = map2d(&mk, a.kring, a.hd, (uint64_t)a.Hkv * a.R, a.hd, BN);
  if (!rc) rc = map2d(&mv, a.vring, a.hd, (uint64_t)a.Hkv * a.R, a.hd, BN);
  // the dq kernel's key/value blocks: DQ_BN rows (R is a multiple of 128,
  // so a block never wraps around the ring)
  if (!rc) rc = map2d(&mk128, a.kring, a.hd, (uint64_t)a.Hkv * a.R, a.hd, DQ_BN);
  if (!rc) rc = map2d(&mv128, a.vring, a.hd, (uint64_t)a.Hkv * a.R, a.hd, DQ_BN);
  if (rc) return rc;
  static std::atomic<uint64_t> attr_dq{0}, attr_dkv{0};
  {
    cudaError_t e = raise_smem_limit(attr_dq, attn_dq_tc_kernel<NA>, DQ::SMEM);
    if (e == cudaSuccess) e = raise_smem_limit(attr_dkv, attn_dkv_tc_kernel<NA>, DKV::SMEM);
    if (e != cudaSuccess) return (int)e;
  }
  BwdParams p;
  p.n = a.n;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.hd = a.hd;
  p.W = a.W;
  p.R = a.R;
  p.pos0 = a.pos0;
  p.scale = 1.0f / sqrtf((float)a.hd);
  p.scale_log2 = 1.4426950408889634f * p.scale;
  p.lse = a.lse;
  p.dsum = a.Dsum;
  p.ld_lse = a.ld_lse;
  p.dqkv = (bf16*)a.dqkv;
  p.ldg = (int64_t)(a.H + 2 * a.Hkv) * a.hd;
  p.ws = a.ws;
  p.err = err;
  p.cs = a.rope_cs;
  {
    const int warps = a.n * a.H;
    launch_k(attn_bwd_prep_tc_kernel, (warps + 7) / 8, 256, 0, st, (const bf16*)a.dout, (const bf16*)a.out, a.n, a.H,
                                                             a.hd, a.Dsum, a.ld_lse);
  }
  p.parts = split_parts(a, num_sms, BM, DQ_BN, 4, 0.02);
  const int64_t plane = (int64_t)a.n * a.H * a.hd;
  while (p.parts > 1 && (int64_t)p.parts * plane > a.ws_elems) --p.parts;
  // dk / dv beside dq on a.side when the scratch holds its two planes after
  // dq's parts (the two kernel pairs share only the prep's D and write
  // disjoint columns of dqkv)
  const int dq_planes = p.parts > 1 ? p.parts : 0;
  const bool beside = a.side && a.side_ev[0] && a.side_ev[1] && (int64_t)(dq_planes + 2) * plane <= a.ws_elems;
  cudaStream_t sk = beside ? a.side : st;
  BwdParams pk = p;
  if (beside) {
    pk.ws = a.ws + (int64_t)dq_planes * plane;
    cudaEventRecord(a.side_ev[0], st);
    cudaStreamWaitEvent(a.side, a.side_ev[0], 0);
  }
  launch_k(attn_dq_tc_kernel<NA>, dim3((a.n + BM - 1) / BM, a.H, p.parts), 576, DQ::SMEM, st, mq, mdo, mk128, mv128,
                                                                                        p);
  if (p.parts > 1) {
    const int cols = a.H * a.hd;
    const int64_t quads = plane / 4;
    const int grid = (int)std::min<int64_t>((quads + 255) / 256, (int64_t)num_sms * 8);
    launch_k(attn_dq_reduce_kernel, grid, 256, 0, st, a.ws, p.parts, a.n, cols, p.dqkv, p.ldg, p.cs, a.hd);
  }
  // dk / dv: beside dq, or after the dq reduction (which may then use the
  // same scratch)
  launch_k(attn_dkv_tc_kernel<NA>, dim3(a.H, (a.n + BM - 1) / BM), 320, DKV::SMEM, sk, mq64, mdo64, mk, mv, pk);
  {
    const int64_t quads = (int64_t)2 * a.n * a.Hkv * a.hd / 4;
    const int grid = (int)std::min<int64_t>((quads + 255) / 256, (int64_t)num_sms * 8);
    launch_k(attn_dkv_reduce_kernel, grid, 256, 0, sk, pk.ws, a.n, a.H, a.Hkv, a.hd, p.dqkv, p.ldg, p.cs);
  }
  if (beside) {
    cudaEventRecord(a.side_ev[1], a.side);
    cudaStreamWaitEvent(st, a.side_ev[1], 0);
  }
  return (int)cudaPeekAtLastError();
}

bool attn_bwd_tc_supported(const AttnArgs& a) {
  return attn_tc_supported(a) && a.pos0 % BN == 0 && ((uintptr_t)a.dout & 15) == 0 &&
         ((uintptr_t)a.dqkv & 15) == 0 && a.ws != nullptr &&
         a.ws_elems >= (int64_t)2 * a.n * a.H * a.hd;
}

int attn_bwd_tc(const AttnArgs& a, int* err, cudaStream_t st) {
  if (a.n <= 0) return 0;
  if (!encoder() || !attn_bwd_tc_supported(a)) return (int)cudaErrorNotSupported;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return a.hd <= 64 ? launch_bwd<1>(a, err, st, sms) : launch_bwd<2>(a, err, st, sms);
}

}  // namespace ttt
