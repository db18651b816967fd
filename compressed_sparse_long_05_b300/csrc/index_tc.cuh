// Lightning-indexer scores on the tcgen05 tensor cores.
//
// DeepSeek-V4 report (Chinese translation, blog.uika.cn) §2.3.1 "Lightning
// Indexer": I[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . K[s,:]); paper notes
// (awesome.papernotes.org) 关键设计 1.  Entry s is visible to query t iff
// (s+1)*m <= t+1; invisible scores are -inf.
//
// Tile: D[128 entries x (QT queries * H heads)] = K_tile[128 x c] * q_group^T,
// one tcgen05.mma chain (M=128, N=QT*H <= 256, K=c in steps of 16), bf16
// operands staged by TMA in 128-byte-swizzled K-major tiles, fp32 accumulators
// double-buffered in tensor memory.  The epilogue reads each entry's row of
// the accumulator (one TMEM lane per entry) and folds the H heads with
// ReLU * w into QT scores per entry: the head reduction never leaves
// registers, and each warp stores 32 consecutive scores per query.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA
// issuer, warps 2-9 epilogue in two groups of four (one warp per TMEM lane
// quarter) that take alternate tiles, so the fold of one tile overlaps the
// next tile's.
//
// Work items are (batch row b, query group g, chunk of entry tiles), dealt
// round-robin to persistent CTAs.  Tiles past the last entry any query of the
// group can see take no MMA: the epilogue writes -inf there directly.
#pragma once
#include "tc.cuh"

namespace csa {

constexpr int IDX_THREADS = 320;
constexpr int IDX_TILE = 128;   // entries per tile (MMA M)

struct IndexTcArgs {
  const float* w;        // [B, Tq, H]
  void* scores;          // [B, Tq, N] float32, or bf16 when scores_bf16
  int scores_bf16;       // 1 = scores rounded to bf16 (the histogram counts the rounded values)
  const int32_t* q_pos;  // [B, Tq] query positions (null: t = i)
  int B, Tq, N, m;
  int QT;                // queries per group (QT * H <= 256)
  int G;                 // query groups per batch row
  int tiles_max;         // ceil(N / 128)
  int stages;            // K-tile pipeline stages (bf16 kernel)
  int chunk_tiles;       // entry tiles per work item
  int chunks;            // work items per group
  int items;             // B * G * chunks
  uint32_t tmem_cols;    // allocated TMEM columns (power of 2 >= nbuf * QT * H)
  int nbuf;              // accumulator buffers in tensor memory (2 or 4)
  uint32_t* hist;        // optional [B * Tq][IDX_HBINS] key-digit histograms (QT == 1), zeroed
  RowPages k_pg;         // paged keys: the K map spans {c, block_rows, num_blocks} (no table: flat)
  int k_piece;           // paged keys: rows per TMA copy, min(block_rows, 128)
  // Failure-detection test hooks (zero in every normal launch):
  unsigned long long wait_ns;   // limit of every wait in ns (0: WAIT_LIMIT_NS)
  int skip_load_plus1;          // n > 0: CTA 0's producer leaves out its K-tile copy number n-1
};

// Key-digit histogram of the scores, built in the index epilogue for the
// top-k selector: bin = top IDX_HBITS bits of the order-preserving key.
constexpr int IDX_HBITS = 11;
constexpr int IDX_HBINS = 1 << IDX_HBITS;

// Paged keys: entry tile j of batch row b arrives as IDX_TILE / k_piece TMA
// copies, copy q from the block that holds logical rows j*IDX_TILE + q*k_piece
// onwards.  key_block gives that block, or -1 when the copy is left out: its
// logical block lies past the sequence's keys (those rows are not visible, so
// their scores are never stored as computed), or the table names a block
// outside the pool (flagged when `flag`).
CSA_DEVINL int key_block(const IndexTcArgs& a, int b, int j, int q, bool flag) {
  // block_rows is a power of two for paged keys: shifts, 32-bit (N < 2^31)
  const int sh = a.k_pg.shift;
  const unsigned int lb = ((unsigned int)j * IDX_TILE + (unsigned int)(q * a.k_piece)) >> sh;
  if (lb >= (((unsigned int)a.N + (1u << sh) - 1u) >> sh)) return -1;
  const int blk = __ldg(a.k_pg.table + (size_t)b * a.k_pg.max_blocks + lb);
  if (blk < 0 || blk >= a.k_pg.num_blocks) {
    if (flag) csa_flag_error(ERRBIT_BAD_INDEX);
    return -1;
  }
  return blk;
}
// Row offset of tile j inside its block (nonzero only when block_rows > IDX_TILE).
CSA_DEVINL int key_block_off(const IndexTcArgs& a, int j) {
  return (int)(((unsigned int)j * IDX_TILE) & ((1u << a.k_pg.shift) - 1u));
}

// Store one score (float32, or rounded to bf16) at element e of the score rows.
CSA_DEVINL void store_score(void* scores, int bf16, size_t e, float v) {
  if (bf16) reinterpret_cast<__nv_bfloat16*>(scores)[e] = __float2bfloat16_rn(v);
  else reinterpret_cast<float*>(scores)[e] = v;
}
// The value a stored score holds (bf16 scores: the rounded value), for the histogram.
CSA_DEVINL float stored_score(int bf16, float v) {
  return bf16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

// One warp's visible scores of one tile into its shared histogram.
CSA_DEVINL void hist_add(uint32_t* wh, float score, bool visible) {
  const uint32_t am = __ballot_sync(0xffffffffu, visible);
  if (visible) {
    const uint32_t dig = float_to_key(score) >> (32 - IDX_HBITS);
    const uint32_t peers = __match_any_sync(am, dig);
    if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(wh + dig, (uint32_t)__popc(peers));
  }
}
// The eight epilogue warps (thread e of 256) add the four per-quarter shared
// histograms into the row's global one and clear them: one global atomic per
// nonzero bin of the CTA, eight bins per thread.
CSA_DEVINL void hist_flush(uint32_t* h4, uint32_t* gh, int e) {
#pragma unroll
  for (int b = e; b < IDX_HBINS; b += 256) {
    const uint32_t c = h4[b] + h4[IDX_HBINS + b] + h4[2 * IDX_HBINS + b] + h4[3 * IDX_HBINS + b];
    if (c) {
      atomicAdd(gh + b, c);
      h4[b] = 0;
      h4[IDX_HBINS + b] = 0;
      h4[2 * IDX_HBINS + b] = 0;
      h4[3 * IDX_HBINS + b] = 0;
    }
  }
}

// Shared-memory layout, sized at launch: S K-tile stages (4, or 6 when the
// query group is at most 64 rows), the query group, head weights, barriers.
template <int H, int C>
struct IndexSmem {
  static constexpr int MAX_STAGES = 6;
  static constexpr int A_BYTES = IDX_TILE * C * 2;       // one K tile
  static constexpr int KCH = C / 64;                     // 64-element swizzle chunks along c
  static constexpr int HIST_BYTES = 4 * IDX_HBINS * 4;   // one histogram per epilogue warp
  int S, OFF_B, OFF_W, OFF_HIST, OFF_BAR, BYTES;
  __host__ __device__ IndexSmem(int stages, int nqh, bool hist) {
    S = stages;
    OFF_B = S * A_BYTES;
    OFF_W = OFF_B + ((nqh * C * 2 + 1023) & ~1023);      // float w_s[8 warps][256]
    OFF_HIST = OFF_W + 8 * 256 * 4;
    OFF_BAR = OFF_HIST + (hist ? HIST_BYTES : 0);
    BYTES = OFF_BAR + 256 + 1024;                        // + alignment slack
  }
  static int stages_for(int nqh, bool hist) {
    for (int s = MAX_STAGES; s > 4; --s)
      if (IndexSmem(s, nqh, hist).BYTES <= 224 * 1024) return s;
    return 4;
  }
};

CSA_DEVINL int vis_of(long long t, int m, int N) {
  if (t < 0) return 0;
  long long v = (t + 1) / m;
  return (int)(v < N ? v : N);
}

// Fold the H accumulator columns of one query in this warp's 32 TMEM lanes:
// sum_h w[h] * ReLU(D[lane][h]).  Two 32-column loads in flight before each
// wait, four independent partial sums (the head reduction is a tree, not a
// 64-deep dependency chain).
template <int H>
CSA_DEVINL float fold_heads(uint32_t taddr, const float* wq) {
  float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
  for (int h0 = 0; h0 < H; h0 += 64) {
    constexpr int kMax = 64;
    const int nh = (H - h0) < kMax ? (H - h0) : kMax;
    uint32_t r[64];
    tmem_ld32(taddr + h0, r);
    if (nh > 32) tmem_ld32(taddr + h0 + 32, r + 32);
    tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < nh; h += 4) {
      const float4 w4 = *reinterpret_cast<const float4*>(wq + h0 + h);
      p0 = fmaf(w4.x, fmaxf(__uint_as_float(r[h]), 0.f), p0);
      p1 = fmaf(w4.y, fmaxf(__uint_as_float(r[h + 1]), 0.f), p1);
      p2 = fmaf(w4.z, fmaxf(__uint_as_float(r[h + 2]), 0.f), p2);
      p3 = fmaf(w4.w, fmaxf(__uint_as_float(r[h + 3]), 0.f), p3);
    }
  }
  return (p0 + p1) + (p2 + p3);
}

struct IdxItem {
  int b, g, t0, nq, j0, j1, jv;   // tiles [j0, j1) of the chunk; MMA for j < jv
};

// visible entries of query row t0 + qi of item x (a negative position sees nothing)
CSA_DEVINL int item_vis(const IndexTcArgs& a, const IdxItem& x, int qi) {
  const long long t = query_pos(a.q_pos, (long long)x.b * a.Tq + x.t0 + qi, x.t0 + qi);
  return vis_of(t, a.m, a.N);
}
// Flags a negative query position of item x (called by one lane per item).
CSA_DEVINL void check_item_pos(const IndexTcArgs& a, const IdxItem& x) {
  for (int qi = 0; qi < x.nq; ++qi)
    if (query_pos(a.q_pos, (long long)x.b * a.Tq + x.t0 + qi, x.t0 + qi) < 0)
      csa_flag_error(ERRBIT_BAD_INDEX);
}

// Tiles [j0, j1) of item `it` (its chunk of the entry range), which do not
// depend on the query positions.
CSA_DEVINL void idx_chunk(const IndexTcArgs& a, int it, int& b, int& j0, int& j1) {
  b = it / (a.G * a.chunks);
  const int c = (it % (a.G * a.chunks)) % a.chunks;
  j0 = c * a.chunk_tiles;
  j1 = min(a.tiles_max, j0 + a.chunk_tiles);
}

CSA_DEVINL IdxItem idx_item(const IndexTcArgs& a, int it) {
  IdxItem x;
  x.b = it / (a.G * a.chunks);
  const int rem = it % (a.G * a.chunks);
  x.g = rem / a.chunks;
  const int c = rem % a.chunks;
  x.t0 = x.g * a.QT;
  x.nq = min(a.QT, a.Tq - x.t0);
  int vis_max = 0;                               // the group's widest query decides the MMA tiles
  for (int qi = 0; qi < x.nq; ++qi) vis_max = max(vis_max, item_vis(a, x, qi));
  const int tiles_vis = (vis_max + IDX_TILE - 1) / IDX_TILE;
  x.j0 = c * a.chunk_tiles;
  x.j1 = min(a.tiles_max, x.j0 + a.chunk_tiles);
  x.jv = max(x.j0, min(x.j1, tiles_vis));
  return x;
}

template <int H, int C>
__global__ void __launch_bounds__(IDX_THREADS, 1)
index_tc_kernel(const __grid_constant__ CUtensorMap tm_K, const __grid_constant__ CUtensorMap tm_q,
                IndexTcArgs a) {
  const int NQH = a.QT * H;                      // MMA N
  const uint64_t lim = a.wait_ns ? a.wait_ns : WAIT_LIMIT_NS;
  const IndexSmem<H, C> L(a.stages, NQH, a.hist != nullptr);
  const int S = L.S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem<1024>(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + L.OFF_B;
  float* w_s = reinterpret_cast<float*>(smem + L.OFF_W);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.OFF_BAR);
  uint64_t* full = bars;                         // [MAX_STAGES]
  uint64_t* empty = bars + L.MAX_STAGES;         // [MAX_STAGES]
  uint64_t* acc_full = bars + 2 * L.MAX_STAGES;  // [nbuf <= 4]
  uint64_t* acc_empty = acc_full + 4;            // [nbuf <= 4]
  uint64_t* b_full = acc_empty + 4;
  uint64_t* b_free = b_full + 1;
  uint64_t* mma_done = b_free + 1;
  uint64_t* epi_sync = mma_done + 1;             // the 8 epilogue warps at an item's end (count 8)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_sync + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t B_BYTES = (uint32_t)NQH * C * 2;
  if (threadIdx.x == 0) { CSA_TRACE_WALL(32); CSA_TRACE_MARK(33); }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
    for (int s = 0; s < 4; ++s) { mbar_init(acc_full + s, 1); mbar_init(acc_empty + s, 4); }
    mbar_init(b_full, 1);
    mbar_init(b_free, 1);
    mbar_init(mma_done, 1);
    mbar_init(epi_sync, 8);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, a.tmem_cols);
    tmem_relinquish();
  }
  if (a.hist) {
    uint32_t* h = reinterpret_cast<uint32_t*>(smem + L.OFF_HIST);
    for (int b = threadIdx.x; b < 4 * IDX_HBINS; b += blockDim.x) h[b] = 0;
  }
  if (warp == 0 && lane == 0) { prefetch_tmap(&tm_K); prefetch_tmap(&tm_q); }
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
      auto load_a = [&](int b, int j) -> bool {
          const uint32_t st = ia % S, ph = (ia / S) & 1;
          if (!mbar_wait(empty + st, ph ^ 1, abort_flag, lim)) return false;
          if (blockIdx.x == 0 && a.skip_load_plus1 == (int)ia + 1) {
            ++ia;          // test hook: this stage never fills, its consumer's wait runs out
            return true;
          }
          if (a.k_pg.table) {
            // paged keys: one copy per k_piece rows from its own block
            const int np = IDX_TILE / a.k_piece, off = key_block_off(a, j);
            uint32_t mask = 0;
            for (int q = 0; q < np; ++q)
              if (key_block(a, b, j, q, true) >= 0) mask |= 1u << q;
            mbar_arrive_expect_tx(full + st, (uint32_t)(__popc(mask) * a.k_piece * 128 * L.KCH));
            for (int q = 0; q < np; ++q) {
              if (!(mask >> q & 1u)) continue;
              const int blk = key_block(a, b, j, q, false);
              for (int kc = 0; kc < L.KCH; ++kc)
                tma_load_3d(sA + st * L.A_BYTES + kc * (IDX_TILE * 128) + q * a.k_piece * 128, &tm_K,
                            full + st, kc * 64, off, blk);
            }
            ++ia;
            return true;
          }
          mbar_arrive_expect_tx(full + st, L.A_BYTES);
#pragma unroll
          for (int kc = 0; kc < L.KCH; ++kc)
            tma_load_3d(sA + st * L.A_BYTES + kc * (IDX_TILE * 128), &tm_K, full + st, kc * 64,
                        j * IDX_TILE, b);
          ++ia;
          return true;
        };
      for (int it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
        // The CTA's first item: its first S tiles go out before the query
        // positions are read (the copies do not depend on them), so the position
        // read overlaps them.  Tiles that turn out invisible are waited out and
        // released by the MMA warp.
        int spec = 0;
        if (it == (int)blockIdx.x) {
          int b0, j0, j1;
          idx_chunk(a, it, b0, j0, j1);
          spec = max(0, min(S, j1 - j0));
          for (int jj = 0; jj < spec && ok; ++jj) {
            ok = load_a(b0, j0 + jj);
            if (jj == 0) CSA_TRACE_MARK(46);
          }
          if (!ok) break;
        }
        const IdxItem x = idx_item(a, it);
        if (nitem == 0) CSA_TRACE_MARK(45);
        if (x.jv <= x.j0) continue;
        const int ntl = x.jv - x.j0;
        // prefetch the first tiles of this item, then swap in its query group
        const int pre = max(spec, min(ntl, S));
        for (int jj = spec; jj < pre && ok; ++jj) ok = load_a(x.b, x.j0 + jj);
        if (nitem == 0) CSA_TRACE_MARK(47);
        if (!ok) break;
        if (nitem > 0 && !mbar_wait(b_free, (nitem - 1) & 1, abort_flag, lim)) { ok = false; break; }
        mbar_arrive_expect_tx(b_full, B_BYTES);
        for (int kc = 0; kc < L.KCH; ++kc)
          tma_load_3d(sB + kc * (NQH * 128), &tm_q, b_full, kc * 64, x.t0 * H, x.b);
        b_issued = true;
        if (nitem == 0) CSA_TRACE_MARK(35);
        ++nitem;
        for (int jj = pre; jj < ntl && ok; ++jj) ok = load_a(x.b, x.j0 + jj);
      }
      // drain copies still in flight before the CTA may exit
      for (uint32_t k = (ia > (uint32_t)S ? ia - S : 0); k < ia; ++k)
        mbar_drain(full + (k % S), (k / S) & 1, lim);
      if (b_issued) mbar_drain(b_full, (nitem - 1) & 1, lim);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t ia = 0, iacc = 0, nitem = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16(IDX_TILE, NQH);
      for (int it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
        const IdxItem x = idx_item(a, it);
        // first item: stages the producer filled ahead for tiles past the visible ones
        const int extra = it == (int)blockIdx.x
                              ? max(0, max(0, min(S, x.j1 - x.j0)) - max(0, x.jv - x.j0)) : 0;
        if (x.jv > x.j0) {
          if (!mbar_wait(b_full, nitem & 1, abort_flag, lim)) { ok = false; break; }
          for (int j = x.j0; j < x.jv; ++j) {
            const uint32_t st = ia % S, ph = (ia / S) & 1;
            const uint32_t buf = iacc % a.nbuf, aph = (iacc / a.nbuf) & 1;
            if (!mbar_wait(acc_empty + buf, aph ^ 1, abort_flag, lim)) { ok = false; break; }
            if (!mbar_wait(full + st, ph, abort_flag, lim)) { ok = false; break; }
            if (ia == 0) CSA_TRACE_MARK(36);
            tc_fence_after();
            const uint32_t aBase = smem_u32(sA + st * L.A_BYTES);
            const uint32_t bBase = smem_u32(sB);
            const uint32_t d = tmem + buf * (uint32_t)NQH;
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk) {
              const uint32_t kc = kk / 4, ko = (kk % 4) * 32;
              const uint64_t ad = sdesc_sw128(aBase + kc * (IDX_TILE * 128) + ko, 16, 1024);
              const uint64_t bd = sdesc_sw128(bBase + kc * (NQH * 128) + ko, 16, 1024);
              umma_f16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
            }
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
        for (int e = 0; e < extra; ++e, ++ia) {     // no MMA reads them: wait for the copy, release
          const uint32_t st = ia % S, ph = (ia / S) & 1;
          if (!mbar_wait(full + st, ph, abort_flag, lim)) { ok = false; break; }
          mbar_arrive(empty + st);
        }
      }
      umma_commit(mma_done);
      mbar_drain(mma_done, 0, lim);
    }
  } else {
    // ---------------- epilogue (warps 2..9: two groups, alternate tiles) ----------------
    const int ew = warp - 2;                       // 0..7
    const int grp = ew >> 2;                       // tiles with iacc % 2 == grp
    const int q4 = warp & 3;                       // TMEM lane quarter of this warp
    uint32_t* wh = reinterpret_cast<uint32_t*>(smem + L.OFF_HIST) + q4 * IDX_HBINS;   // shared by both groups
    uint32_t iacc = 0, nsync = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
      const IdxItem x = idx_item(a, it);
      // this warp's own copy of the group's head weights (no cross-warp barrier,
      // so a warp that stops on a timed-out wait cannot strand the others)
      float* ws = w_s + ew * 256;
      if (ew == 0 && lane == 0 && x.j0 == 0) check_item_pos(a, x);
      __syncwarp();                                // the previous item's reads are done
      for (int e = lane; e < x.nq * H; e += 32)
        ws[e] = __ldg(a.w + ((size_t)x.b * a.Tq + x.t0) * H + e);
      __syncwarp();
      for (int j = x.j0; j < x.j1; ++j) {
        const int s = j * IDX_TILE + q4 * 32 + lane;
        const size_t srow = ((size_t)x.b * a.Tq + x.t0) * a.N + s;   // element of this lane's first score
        if (j < x.jv) {
          const uint32_t mine = (iacc & 1) == (uint32_t)grp;
          const uint32_t buf = iacc % a.nbuf, aph = (iacc / a.nbuf) & 1;
          ++iacc;
          if (!mine) continue;
          if (!mbar_wait(acc_full + buf, aph, abort_flag, lim)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tbase = tmem + ((uint32_t)(q4 * 32) << 16) + buf * (uint32_t)NQH;
          for (int qi = 0; qi < x.nq; ++qi) {
            const float acc = fold_heads<H>(tbase + qi * H, ws + qi * H);
            const int vis = item_vis(a, x, qi);
            if (s < a.N) store_score(a.scores, a.scores_bf16, srow + (size_t)qi * a.N, s < vis ? acc : -INFINITY);
            if (a.hist) hist_add(wh, stored_score(a.scores_bf16, acc), s < vis);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty + buf);
          if (ew == 0 && lane == 0) CSA_TRACE_MARK(iacc <= 2 ? 38 : 39);
        } else if ((j & 1) == grp) {
          for (int qi = 0; qi < x.nq; ++qi)
            if (s < a.N) store_score(a.scores, a.scores_bf16, srow + (size_t)qi * a.N, -INFINITY);
        }
      }
      if (ew == 0 && lane == 0) CSA_TRACE_MARK(40);
      if (a.hist) {
        // both groups have added this item's scores: all eight warps flush (and
        // clear) the shared per-quarter histograms; the next item's adds wait for that.
        // Bounded waits: a warp that gave up still arrives, and the flag ends the rest.
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_sync);
        const bool s1 = __all_sync(0xffffffffu, mbar_wait(epi_sync, nsync & 1, abort_flag, lim));
        ++nsync;
        if (ew == 0 && lane == 0) CSA_TRACE_MARK(41);
        if (ok && s1)
          hist_flush(reinterpret_cast<uint32_t*>(smem + L.OFF_HIST),
                     a.hist + ((size_t)x.b * a.Tq + x.t0) * IDX_HBINS, ew * 32 + lane);
        if (ew == 0 && lane == 0) CSA_TRACE_MARK(42);
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_sync);
        const bool s2 = __all_sync(0xffffffffu, mbar_wait(epi_sync, nsync & 1, abort_flag, lim));
        ++nsync;
        if (!s1 || !s2) ok = false;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, a.tmem_cols);
  if (threadIdx.x == 0) { CSA_TRACE_MARK(44); CSA_TRACE_WALL(43); }
}

}  // namespace csa
