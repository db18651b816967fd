// Grouped output projection on the tcgen05 tensor cores.
//
// DeepSeek-V4 report (Chinese translation, blog.uika.cn) §2.3.1 "分组输出投影":
// c * n_h is large, so the n_h head outputs are split into g groups, each group
// is projected to a d_g-dimensional intermediate output, and the g outputs are
// then projected to the model width d (§4.2.1: V4-Pro g = 16, d_g = 1024,
// d = 7168; V4-Flash g = 8, d_g = 1024, d = 4096).
//
// Both projections are one kernel: for each group j < G,
//     C[:, j*N : (j+1)*N] = A[:, j*K : (j+1)*K] * W_j^T
// with A [M rows, stride lda] and C [M rows, stride ldc] bf16 row-major, W
// [G, N, K] bf16 (each group's weight stored output-major, i.e. K-major, as
// the MMA reads it), fp32 accumulation, bf16 result.  The grouped step has
// G = g, K = (n_h / g) * c, N = d_g; the final step G = 1, K = g * d_g, N = d.
//
// Tiles of 128 x 256 outputs, K in steps of 64 (one 128-byte swizzle atom):
// warp 0 issues TMA loads of A [128 x 64] (tensor map dims {K, G, M}, so
// every stride grows outward) and W [256 x 64] into a 4-stage
// ring, warp 1 owns tensor memory and issues tcgen05.mma (M = 128, N = 256,
// K = 16) from one thread into one of two accumulators (256 columns each),
// warps 2-5 drain the other accumulator (one TMEM lane quarter each: a thread
// owns one output row) and store bf16.  Persistent CTAs walk the tiles in
// super-rows of GM M-blocks: all N-blocks of GM M-blocks run before the next
// GM, so the A rows being reused stay in L2 while the weights stream.
#pragma once
#include "tc.cuh"

namespace csa {

constexpr int GEMM_THREADS = 192;
constexpr int GEMM_BM = 128, GEMM_BN = 256, GEMM_BK = 64;
constexpr int GEMM_STAGES = 4;
constexpr int GEMM_GM = 16;             // M-blocks per raster super-row

struct GemmSmem {
  static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;     // 16 KB
  static constexpr int B_BYTES = GEMM_BN * GEMM_BK * 2;     // 32 KB
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int OFF_BAR = GEMM_STAGES * STAGE;
  static constexpr int BYTES = OFF_BAR + 256 + 1024;        // + alignment slack
};

struct GemmArgs {
  __nv_bfloat16* C;
  long long ldc;          // elements between rows of C
  int M, N, K, G;         // per group: C_j [M x N] = A_j [M x K] * W_j^T
  int MT, NT;             // M- and N-blocks per group
  long long tiles;        // G * MT * NT
  uint64_t wait_ns;       // 0: WAIT_LIMIT_NS
};

struct GemmTile {
  int g, mt, nt;
};

// tile index -> (group, M-block, N-block): groups outermost, then super-rows
// of GEMM_GM M-blocks, N-blocks, M-blocks within the super-row innermost
CSA_DEVINL GemmTile gemm_tile(const GemmArgs& a, long long t) {
  GemmTile x;
  const long long per_g = (long long)a.MT * a.NT;
  x.g = (int)(t / per_g);
  long long r = t % per_g;
  const long long sup_len = (long long)GEMM_GM * a.NT;
  const int sup = (int)(r / sup_len);
  r %= sup_len;
  const int gm = min(GEMM_GM, a.MT - sup * GEMM_GM);   // M-blocks in this super-row
  x.nt = (int)(r / gm);
  x.mt = sup * GEMM_GM + (int)(r % gm);
  return x;
}

__global__ void __launch_bounds__(GEMM_THREADS, 1)
gemm_grouped_kernel(const __grid_constant__ CUtensorMap tm_A, const __grid_constant__ CUtensorMap tm_W,
                    const GemmArgs a) {
  using L = GemmSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem<1024>(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* full = bars;                           // [STAGES] A + W tile landed
  uint64_t* empty = bars + GEMM_STAGES;            // [STAGES] MMAs that read the stage done
  uint64_t* acc_full = bars + 2 * GEMM_STAGES;     // [2] accumulator complete
  uint64_t* acc_empty = acc_full + 2;              // [2] epilogue drained it (count 4)
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint64_t lim = a.wait_ns ? a.wait_ns : WAIT_LIMIT_NS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = (a.K + GEMM_BK - 1) / GEMM_BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < GEMM_STAGES; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(acc_full + s, 1); mbar_init(acc_empty + s, 4); }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) { prefetch_tmap(&tm_A); prefetch_tmap(&tm_W); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_enter();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (long long t = blockIdx.x; t < a.tiles && ok; t += gridDim.x) {
        const GemmTile x = gemm_tile(a, t);
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const uint32_t st = it % GEMM_STAGES, ph = (it / GEMM_STAGES) & 1;
          if (!mbar_wait(empty + st, ph ^ 1, abort_flag, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(full + st, L::STAGE);
          uint8_t* sA = smem + st * L::STAGE;
          tma_load_3d(sA, &tm_A, full + st, ks * GEMM_BK, x.g, x.mt * GEMM_BM);
          tma_load_3d(sA + L::A_BYTES, &tm_W, full + st, ks * GEMM_BK, x.nt * GEMM_BN, x.g);
        }
      }
      // drain copies still in flight before the CTA may exit
      for (uint32_t k = (it > (uint32_t)GEMM_STAGES ? it - GEMM_STAGES : 0); k < it; ++k)
        mbar_drain(full + (k % GEMM_STAGES), (k / GEMM_STAGES) & 1, lim);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(GEMM_BM, GEMM_BN);
      uint32_t it = 0, nt = 0;
      bool ok = true;
      for (long long t = blockIdx.x; t < a.tiles && ok; t += gridDim.x, ++nt) {
        const uint32_t buf = nt & 1, aph = (nt >> 1) & 1;
        if (!mbar_wait(acc_empty + buf, aph ^ 1, abort_flag, lim)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + buf * GEMM_BN;
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const uint32_t st = it % GEMM_STAGES, ph = (it / GEMM_STAGES) & 1;
          if (!mbar_wait(full + st, ph, abort_flag, lim)) { ok = false; break; }
          tc_fence_after();
          const uint32_t aBase = smem_u32(smem + st * L::STAGE);
          const uint32_t bBase = aBase + L::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < GEMM_BK / 16; ++kk)
            umma_f16(d, sdesc_sw128(aBase + kk * 32, 16, 1024), sdesc_sw128(bBase + kk * 32, 16, 1024),
                     idesc, (ks | kk) ? 1u : 0u);
          umma_commit(empty + st);
        }
        if (!ok) break;
        umma_commit(acc_full + buf);
      }
      umma_commit(mma_done);
      mbar_drain(mma_done, 0, lim);
    }
  } else {
    // ---------------- epilogue (warps 2-5) ----------------
    const int q4 = warp & 3;                       // TMEM lane quarter this warp may read
    uint32_t nt = 0;
    for (long long t = blockIdx.x; t < a.tiles; t += gridDim.x, ++nt) {
      const GemmTile x = gemm_tile(a, t);
      const uint32_t buf = nt & 1, aph = (nt >> 1) & 1;
      if (!mbar_wait(acc_full + buf, aph, abort_flag, lim)) break;
      tc_fence_after();
      const int row = x.mt * GEMM_BM + q4 * 32 + lane;
      const int col0 = x.nt * GEMM_BN;
      __nv_bfloat16* crow = a.C + (size_t)row * a.ldc + (size_t)x.g * a.N + col0;
      const uint32_t tbase = tmem + ((uint32_t)(q4 * 32) << 16) + buf * GEMM_BN;
#pragma unroll 1
      for (int c = 0; c < GEMM_BN; c += 64) {
        uint32_t r[64];
        tmem_ld32(tbase + c, r);
        tmem_ld32(tbase + c + 32, r + 32);
        tmem_ld_wait();
        if (row < a.M) {
          if (col0 + c + 64 <= a.N) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(r[8 * u + e]);
              *reinterpret_cast<uint4*>(crow + c + 8 * u) = f_to_bf16x8(f);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (col0 + c + e < a.N) crow[c + e] = __float2bfloat16_rn(__uint_as_float(r[e]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + buf);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace csa
