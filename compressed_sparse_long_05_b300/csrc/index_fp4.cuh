// Lightning-indexer scores from FP4 indexer queries and keys, on the tcgen05
// block-scaled tensor path (kind::mxf4nvf4).
//
// DeepSeek-V4 report (Chinese translation, blog.uika.cn) §2.3.4 "效率讨论":
// the lightning indexer's QK runs in FP4; §2.3.1 "Lightning Indexer" defines
// I[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . K[s,:]).  Storage: e2m1 values two
// per byte (element 2j in the low nibble of byte j) times one e4m3 scale per
// 16 consecutive elements, which is exactly the operand format of the
// block-scaled MMA (16-element blocks, ue4m3 scales, scale_vec::4X): the
// products are formed by the tensor cores from the stored bytes, never
// dequantised in memory.
//
// Tile: D[128 entries x (QT*H <= 128)] = K_tile[128 x 128] * q_group^T, as two
// MMAs of K = 64.  Operands are TMA-staged 64-byte-swizzled K-major tiles (one
// 64-byte row per entry).  Scale factors go global -> shared (TMA, as raw
// [rows][8] bytes) -> rearranged by the MMA warp into the 512-byte
// tensor-memory scale atoms (row r = 32g + i of a 128-row block at byte
// 16 i + 4 g + k for the k-th 16-element block of the MMA's K range) ->
// tcgen05.cp into tensor memory (32x128b, replicated to the four lane
// quarters).  fp32 accumulators rotate through up to four tensor-memory
// buffers; the epilogue folds the heads with ReLU * w exactly as the bf16
// kernel does.
//
// Warp roles (384 threads), each step of the per-tile chain on its own warps so
// that no step's latency sits inside another's loop:
//   warp 0      TMA producer (K tile + its scale rows, 12 stages),
//   warp 1      TMEM owner; one lane issues the MMAs,
//   warps 2, 3  scale rearrangement (raw rows -> atoms -> tcgen05.cp into
//               tensor memory) of alternate tiles, running ahead of the MMA,
//   warps 4-11  epilogue, two groups of four warps (one per TMEM lane
//               quarter) taking alternate tiles.
#pragma once
#include "index_tc.cuh"

namespace csa {

constexpr int FP4_STAGES = 12;
constexpr int FP4_THREADS = 384;
constexpr int FP4_EPI_WARP0 = 4;           // first epilogue warp (warps 2, 3 rearrange scales)
constexpr int FP4_C = 128;                  // indexer dim (elements)
constexpr int FP4_ROWB = FP4_C / 2;         // packed bytes per row
constexpr int FP4_SF_BOX = 130;             // uint64 scale rows per stage load (128 + 2 for alignment)

struct IndexFp4Smem {
  static constexpr int A_BYTES = IDX_TILE * FP4_ROWB;        // 8 KB
  static constexpr int RAW_BYTES = FP4_SF_BOX * 8;           // 1040 B
  static constexpr int RAW_PITCH = 1152;
  static constexpr int OFF_A = 0;                            // [STAGES][A_BYTES]
  static constexpr int OFF_B = OFF_A + FP4_STAGES * A_BYTES; // q group, <= 128 rows x 64 B
  static constexpr int OFF_ATOM_A = OFF_B + 128 * FP4_ROWB;  // [STAGES][2][512]
  static constexpr int OFF_ATOM_B = OFF_ATOM_A + FP4_STAGES * 1024;   // [2][512]
  static constexpr int OFF_RAW_A = OFF_ATOM_B + 1024;        // [STAGES][RAW_PITCH]
  static constexpr int OFF_RAW_B = OFF_RAW_A + FP4_STAGES * RAW_PITCH;  // <= 128 x 8 B
  static constexpr int OFF_W = OFF_RAW_B + 1024;             // float w_s[8 warps][2][256]
  static constexpr int OFF_HIST = OFF_W + 8 * 2 * 256 * 4;  // [4 lane quarters][IDX_HBINS] u32
  static constexpr int OFF_BAR = OFF_HIST + 4 * IDX_HBINS * 4;
  static constexpr int NBAR = 3 * FP4_STAGES + 8 + 7;        // stage, accumulator, item barriers
  static constexpr int BAR_BYTES = 512;
  static constexpr int BYTES = OFF_BAR + BAR_BYTES + 1024;   // + alignment slack
  static_assert(NBAR * 8 + 8 <= BAR_BYTES, "barrier region");
};

// Instruction descriptor, kind::mxf4nvf4: A and B e2m1, K-major, ue4m3 scales, D f32.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

CSA_DEVINL void umma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// shared -> tensor memory: 32 rows x 16 bytes, replicated into the 4 lane quarters
CSA_DEVINL void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Shared-memory descriptor of a 64-byte-swizzled K-major tile (64-byte rows,
// 8-row groups 512 B apart).
CSA_DEVINL uint64_t sdesc_sw64(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16 >> 4) << 16;
  d |= (uint64_t)(512 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;   // 64-byte swizzle
  return d;
}
// Descriptor of one 512-byte scale atom (no swizzle, 8-row core matrices 128 B apart).
CSA_DEVINL uint64_t sdesc_atom(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 16;
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// The 32 lanes of a warp turn raw scale rows (8 bytes each, rows [0, nrows))
// into the two 512-byte atoms (K-step 0: bytes 0-3 of each row, K-step 1:
// bytes 4-7).  Rows >= nrows get zero scales.
CSA_DEVINL void build_scale_atoms(const uint8_t* raw, uint8_t* atoms, int nrows, int lane) {
  uint32_t w0[4], w1[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int r = 32 * g + lane;
    uint2 v = make_uint2(0u, 0u);
    if (r < nrows) {
      v.x = *reinterpret_cast<const uint32_t*>(raw + r * 8);
      v.y = *reinterpret_cast<const uint32_t*>(raw + r * 8 + 4);
    }
    w0[g] = v.x;
    w1[g] = v.y;
  }
  *reinterpret_cast<uint4*>(atoms + lane * 16) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
  *reinterpret_cast<uint4*>(atoms + 512 + lane * 16) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
}

struct IndexFp4Args {
  IndexTcArgs t;           // shared work split (QT * H <= 128)
  const uint8_t* k_sf;     // paged keys: the scale-byte pool (8 bytes per key row)
};

template <int H>
__global__ void __launch_bounds__(FP4_THREADS, 1)
index_fp4_kernel(const __grid_constant__ CUtensorMap tm_K, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_Ksf, const __grid_constant__ CUtensorMap tm_qsf,
                 IndexFp4Args fa) {
  using L = IndexFp4Smem;
  const IndexTcArgs& a = fa.t;
  if (threadIdx.x == 0) { CSA_TRACE_WALL(32); CSA_TRACE_MARK(33); }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem<1024>(smem_raw);
  uint8_t* sA = smem + L::OFF_A;
  uint8_t* sB = smem + L::OFF_B;
  uint8_t* atomA = smem + L::OFF_ATOM_A;
  uint8_t* atomB = smem + L::OFF_ATOM_B;
  uint8_t* rawA = smem + L::OFF_RAW_A;
  uint8_t* rawB = smem + L::OFF_RAW_B;
  float* w_s = reinterpret_cast<float*>(smem + L::OFF_W);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* full = bars;                          // [STAGES] K tile + scale rows landed (TMA)
  uint64_t* sf_ready = bars + FP4_STAGES;         // [STAGES] scale atoms of the stage in tensor memory (commit)
  uint64_t* empty = bars + 2 * FP4_STAGES;        // [STAGES] MMA read the stage (commit)
  uint64_t* acc_full = bars + 3 * FP4_STAGES;     // [nbuf <= 4] accumulator written (commit)
  uint64_t* acc_empty = acc_full + 4;             // [nbuf <= 4] read by the owning epilogue group
  uint64_t* b_full = acc_empty + 4;               // query group + its scale rows landed (TMA)
  uint64_t* b_ready = b_full + 1;                 // query scale atoms in tensor memory (commit)
  uint64_t* b_free = b_ready + 1;                 // every MMA of the item done (commit)
  uint64_t* mma_done = b_free + 1;
  uint64_t* epi_sync = mma_done + 1;              // the 8 epilogue warps at an item's end (count 8)
  uint64_t* cp_done = epi_sync + 1;               // [2] each scale warp's last copies (commit)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cp_done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NQH = a.QT * H;                       // MMA N (<= 128)
  // tensor-memory columns: accumulators [0, nbuf*NQH) within [0, 256), A scales, B scales
  const uint32_t TM_SFA = 256, TM_SFB = 256 + FP4_STAGES * 8;

  if (threadIdx.x == 0) {
    for (int s = 0; s < FP4_STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(sf_ready + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int s = 0; s < 4; ++s) { mbar_init(acc_full + s, 1); mbar_init(acc_empty + s, 4); }
    mbar_init(b_full, 1);
    mbar_init(b_ready, 1);
    mbar_init(b_free, 1);
    mbar_init(mma_done, 1);
    mbar_init(epi_sync, 8);
    mbar_init(cp_done, 1);
    mbar_init(cp_done + 1, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (a.hist) {
    uint32_t* h = reinterpret_cast<uint32_t*>(smem + L::OFF_HIST);
    for (int b = threadIdx.x; b < 4 * IDX_HBINS; b += blockDim.x) h[b] = 0;
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_K); prefetch_tmap(&tm_q); prefetch_tmap(&tm_Ksf); prefetch_tmap(&tm_qsf);
  }
  if (warp == 2 && lane == 0 && (int)blockIdx.x < a.items) {
    // the first item's query positions and head weights
    int b0, j0, j1;
    idx_chunk(a, blockIdx.x, b0, j0, j1);
    const int t0 = ((int)blockIdx.x % (a.G * a.chunks)) / a.chunks * a.QT;
    if (a.q_pos) prefetch_l1(a.q_pos + (size_t)b0 * a.Tq + t0);
    prefetch_l1(a.w + ((size_t)b0 * a.Tq + t0) * H);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_enter();   // barriers and tensor memory are set up; inputs may still be in flight
  if (threadIdx.x == 0) CSA_TRACE_MARK(34);

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t ia = 0, nitem = 0;
      bool ok = true, b_issued = false;
      for (int it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
        const IdxItem x = idx_item(a, it);
        if (x.jv <= x.j0) continue;
        const int ntl = x.jv - x.j0;
        auto load_a = [&](int j) -> bool {
          const uint32_t st = ia % FP4_STAGES, ph = (ia / FP4_STAGES) & 1;
          if (!mbar_wait(empty + st, ph ^ 1, abort_flag)) return false;
          // scale rows of entries j*128 .. j*128+127 of batch row b, from an even
          // (16-byte aligned) flat row index
          if (a.k_pg.table) {
            // paged keys: one K copy and one scale-row copy per k_piece rows from
            // its own block; the scale rows (k_piece * 8 bytes, 64 at the least)
            // come by untiled bulk copy, whose addresses need 16-byte alignment
            // only (a tensor copy's shared destination would need 128), and land
            // from the start of the stage
            const int np = IDX_TILE / a.k_piece, off = key_block_off(a, j);
            uint32_t mask = 0;
            for (int q = 0; q < np; ++q)
              if (key_block(a, x.b, j, q, true) >= 0) mask |= 1u << q;
            mbar_arrive_expect_tx(full + st, (uint32_t)(__popc(mask) * a.k_piece * (FP4_ROWB + 8)));
            for (int q = 0; q < np; ++q) {
              if (!(mask >> q & 1u)) continue;
              const int blk = key_block(a, x.b, j, q, false);
              tma_load_3d(sA + st * L::A_BYTES + q * a.k_piece * FP4_ROWB, &tm_K, full + st, 0, off, blk);
              const size_t sx = (size_t)blk * a.k_pg.block_rows + off;
              bulk_load(rawA + st * L::RAW_PITCH + q * a.k_piece * 8, fa.k_sf + sx * 8,
                        (uint32_t)(a.k_piece * 8), full + st);
            }
            ++ia;
            return true;
          }
          const long long r0 = (long long)x.b * a.N + (long long)j * IDX_TILE;
          const int sx = (int)(r0 & ~1LL);
          mbar_arrive_expect_tx(full + st, L::A_BYTES + L::RAW_BYTES);
          tma_load_3d(sA + st * L::A_BYTES, &tm_K, full + st, 0, j * IDX_TILE, x.b);
          asm volatile(
              "cp.async.bulk.tensor.1d.shared::cluster.global.mbarrier::complete_tx::bytes"
              " [%0], [%1, {%2}], [%3];" ::"r"(smem_u32(rawA + st * L::RAW_PITCH)),
              "l"(reinterpret_cast<uint64_t>(&tm_Ksf)), "r"(sx), "r"(smem_u32(full + st))
              : "memory");
          ++ia;
          return true;
        };
        const int pre = min(ntl, FP4_STAGES);
        for (int jj = 0; jj < pre && ok; ++jj) ok = load_a(x.j0 + jj);
        if (!ok) break;
        if (nitem > 0 && !mbar_wait(b_free, (nitem - 1) & 1, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(b_full, (uint32_t)NQH * (FP4_ROWB + 8));
        tma_load_3d(sB, &tm_q, b_full, 0, x.t0 * H, x.b);
        {
          const int qx = (x.b * a.Tq + x.t0) * H;     // H even: 16-byte aligned
          asm volatile(
              "cp.async.bulk.tensor.1d.shared::cluster.global.mbarrier::complete_tx::bytes"
              " [%0], [%1, {%2}], [%3];" ::"r"(smem_u32(rawB)),
              "l"(reinterpret_cast<uint64_t>(&tm_qsf)), "r"(qx), "r"(smem_u32(b_full))
              : "memory");
        }
        b_issued = true;
        if (nitem == 0) CSA_TRACE_MARK(35);
        ++nitem;
        for (int jj = pre; jj < ntl && ok; ++jj) ok = load_a(x.j0 + jj);
        if (nitem == 1) CSA_TRACE_MARK(59);
      }
      for (uint32_t k = (ia > FP4_STAGES ? ia - FP4_STAGES : 0); k < ia; ++k)
        mbar_drain(full + (k % FP4_STAGES), (k / FP4_STAGES) & 1);
      if (b_issued) mbar_drain(b_full, (nitem - 1) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (one lane) ----------------
    if (lane == 0) {
      uint32_t ia = 0, iacc = 0, nitem = 0;
      bool ok = true;
      const uint32_t idesc = idesc_mxf4(IDX_TILE, NQH);
      const uint32_t bBase = smem_u32(sB);
      for (int it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
        const IdxItem x = idx_item(a, it);
        if (x.jv <= x.j0) continue;
        if (!mbar_wait(b_ready, nitem & 1, abort_flag)) { ok = false; break; }
        for (int j = x.j0; j < x.jv; ++j) {
          const uint32_t st = ia % FP4_STAGES, ph = (ia / FP4_STAGES) & 1;
          const uint32_t buf = iacc % a.nbuf, aph = (iacc / a.nbuf) & 1;
          if (!mbar_wait(acc_empty + buf, aph ^ 1, abort_flag)) { ok = false; break; }
          if (!mbar_wait(sf_ready + st, ph, abort_flag)) { ok = false; break; }
          if (ia == 0) CSA_TRACE_MARK(36);
          tc_fence_after();
          const uint32_t sfa = tmem + TM_SFA + st * 8;
          const uint32_t aBase = smem_u32(sA + st * L::A_BYTES);
          const uint32_t d = tmem + buf * (uint32_t)NQH;
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            umma_mxf4(d, sdesc_sw64(aBase + kk * 32), sdesc_sw64(bBase + kk * 32), idesc,
                      sfa + kk * 4, tmem + TM_SFB + kk * 4, kk > 0 ? 1u : 0u);
          umma_commit(empty + st);
          umma_commit(acc_full + buf);
          ++ia;
          ++iacc;
        }
        if (!ok) break;
        CSA_TRACE_MARK(37);
        umma_commit(b_free);
        ++nitem;
      }
      umma_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else if (warp < FP4_EPI_WARP0) {
    // ---------------- scale rearrangement (whole warps; warp 2 even tiles, warp 3 odd) ----------------
    const uint32_t sw = warp - 2;
    uint32_t ia = 0, nitem = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
      const IdxItem x = idx_item(a, it);
      if (x.jv <= x.j0) continue;
      if (sw == 0) {
        // every lane waits and the warp votes, so all 32 lanes leave together on a timeout
        if (!__all_sync(0xffffffffu, mbar_wait(b_full, nitem & 1, abort_flag))) { ok = false; break; }
        build_scale_atoms(rawB, atomB, NQH, lane);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          // these warps also move the atoms into tensor memory; the commit tells the
          // MMA lane when the copies are done
          tc_fence_after();
          tmem_cp_32x128b_x4(tmem + TM_SFB, sdesc_atom(smem_u32(atomB)));
          tmem_cp_32x128b_x4(tmem + TM_SFB + 4, sdesc_atom(smem_u32(atomB + 512)));
          umma_commit(b_ready);
        }
        __syncwarp();
      }
      for (int j = x.j0; j < x.jv; ++j, ++ia) {
        if ((ia & 1) != sw) continue;
        const uint32_t st = ia % FP4_STAGES, ph = (ia / FP4_STAGES) & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(full + st, ph, abort_flag))) { ok = false; break; }
        const long long r0 = (long long)x.b * a.N + (long long)j * IDX_TILE;
        const uint8_t* raw = rawA + st * L::RAW_PITCH + (a.k_pg.table ? 0 : (r0 & 1) * 8);
        const int nrows = (int)min((long long)IDX_TILE, (long long)a.N - (long long)j * IDX_TILE);
        build_scale_atoms(raw, atomA + st * 1024, nrows, lane);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sfa = tmem + TM_SFA + st * 8;
          tmem_cp_32x128b_x4(sfa, sdesc_atom(smem_u32(atomA + st * 1024)));
          tmem_cp_32x128b_x4(sfa + 4, sdesc_atom(smem_u32(atomA + st * 1024 + 512)));
          umma_commit(sf_ready + st);
          if (sw == 0) CSA_TRACE_MARK(ia == 0 ? 57 : 58);
        }
        __syncwarp();
      }
      ++nitem;
    }
    // every tensor-memory copy this warp issued is done before the CTA frees tensor memory
    if (lane == 0) {
      umma_commit(cp_done + sw);
      mbar_drain(cp_done + sw, 0);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 4..11: two groups, alternate tiles) ----------------
    const int ew = warp - FP4_EPI_WARP0;             // 0..7
    const int grp = ew >> 2;                         // tiles with iacc % 2 == grp
    const int q4 = warp & 3;                         // TMEM lane quarter this warp may access
    uint32_t* wh = reinterpret_cast<uint32_t*>(smem + L::OFF_HIST) + q4 * IDX_HBINS;   // shared by both groups
    uint32_t iacc = 0, nitem = 0, nsync = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
      const IdxItem x = idx_item(a, it);
      float* ws = w_s + ((ew * 2) + (nitem & 1)) * 256;
      if (ew == 0 && lane == 0 && x.j0 == 0) check_item_pos(a, x);
      for (int e = lane; e < x.nq * H; e += 32)
        ws[e] = __ldg(a.w + ((size_t)x.b * a.Tq + x.t0) * H + e);
      __syncwarp();
      ++nitem;
      for (int j = x.j0; j < x.j1; ++j) {
        const int s = j * IDX_TILE + q4 * 32 + lane;
        const size_t srow = ((size_t)x.b * a.Tq + x.t0) * a.N + s;   // element of this lane's first score
        if (j < x.jv) {
          const uint32_t mine = (iacc & 1) == (uint32_t)grp;
          const uint32_t buf = iacc % a.nbuf, aph = (iacc / a.nbuf) & 1;
          ++iacc;
          if (!mine) continue;
          if (ew == 0 && lane == 0 && iacc == 41) CSA_TRACE_MARK(60);   // traced tile
          if (!mbar_wait(acc_full + buf, aph, abort_flag)) { ok = false; break; }
          if (ew == 0 && lane == 0 && iacc == 41) CSA_TRACE_MARK(61);
          tc_fence_after();
          const uint32_t tbase = tmem + ((uint32_t)(q4 * 32) << 16) + buf * (uint32_t)NQH;
          for (int qi = 0; qi < x.nq; ++qi) {
            const float acc = fold_heads<H>(tbase + qi * H, ws + qi * H);
            if (ew == 0 && lane == 0 && iacc == 41) CSA_TRACE_MARK(62);
            const int vis = item_vis(a, x, qi);
            if (s < a.N) store_score(a.scores, a.scores_bf16, srow + (size_t)qi * a.N, s < vis ? acc : -INFINITY);
            if (a.hist) hist_add(wh, stored_score(a.scores_bf16, acc), s < vis);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty + buf);
          if (ew == 0 && lane == 0 && iacc == 41) CSA_TRACE_MARK(63);
          if (ew == 0 && lane == 0) CSA_TRACE_MARK(iacc <= 2 ? 38 : 39);
        } else if ((j & 1) == grp) {
          for (int qi = 0; qi < x.nq; ++qi)
            if (s < a.N) store_score(a.scores, a.scores_bf16, srow + (size_t)qi * a.N, -INFINITY);
        }
      }
      if (a.hist) {
        // both groups have added this item's scores: all eight warps flush (and
        // clear) the shared per-quarter histograms; the next item's adds wait for that.
        // Bounded waits: a warp that gave up still arrives, and the flag ends the rest.
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_sync);
        const bool s1 = __all_sync(0xffffffffu, mbar_wait(epi_sync, nsync & 1, abort_flag));
        ++nsync;
        if (ew == 0 && lane == 0) CSA_TRACE_MARK(41);
        if (ok && s1)
          hist_flush(reinterpret_cast<uint32_t*>(smem + L::OFF_HIST),
                     a.hist + ((size_t)x.b * a.Tq + x.t0) * IDX_HBINS, ew * 32 + lane);
        if (ew == 0 && lane == 0) CSA_TRACE_MARK(42);
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_sync);
        const bool s2 = __all_sync(0xffffffffu, mbar_wait(epi_sync, nsync & 1, abort_flag));
        ++nsync;
        if (!s1 || !s2) ok = false;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0) { CSA_TRACE_MARK(44); CSA_TRACE_WALL(43); }
}

}  // namespace csa
