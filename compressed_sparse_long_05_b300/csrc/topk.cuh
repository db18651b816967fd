// Per-row top-k by exact radix selection (DeepSeek-V4 report, Chinese
// translation blog.uika.cn, §2.3.1 "top-k selector"; paper notes
// awesome.papernotes.org, C_t = TopK_k(I_t,:)).
//
// One thread-block cluster per query row.  The row's visible prefix
// [0, vis) is split into CL contiguous slices, one per CTA, each held in
// shared memory.  Four 8-bit radix passes over order-preserving keys find the
// exact k-th largest key K*: each pass builds per-warp histograms (lanes with
// equal digits aggregated by __match_any_sync), sums them per CTA, and every
// CTA sums the CL CTA histograms through distributed shared memory.  The
// output is every key > K* plus the lowest-index keys == K* needed to reach k,
// written in ascending index order (block scan inside a CTA, cluster prefix
// across CTAs), then -1 padding.  With CL = 1 the same code runs one CTA per
// row (prefill rows).
#pragma once
#include <cooperative_groups.h>
#include "common.cuh"

namespace csa {
namespace cg = cooperative_groups;

constexpr int TOPK_THREADS = 512;
constexpr int TOPK_WARPS = TOPK_THREADS / 32;

struct TopkArgs {
  const float* scores;
  int32_t* idx;
  const int32_t* q_pos;   // [rows] query positions (null: t = i)
  int Tq, N, k, m;
  int slice;   // elements per CTA slice (multiple of 4)
};

// exclusive block scan of one int per thread; returns the total in *total
CSA_DEVINL int block_excl_scan(int x, int* sh_warp, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh_warp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int w = lane < TOPK_WARPS ? sh_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < TOPK_WARPS) sh_warp[lane] = wi - w;   // exclusive warp offsets
    if (lane == TOPK_WARPS - 1) sh_warp[TOPK_WARPS] = wi;
  }
  __syncthreads();
  int res = sh_warp[wid] + incl - x;
  *total = sh_warp[TOPK_WARPS];
  __syncthreads();
  return res;
}

template <int CL>
__global__ void __launch_bounds__(TOPK_THREADS) topk_kernel(TopkArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) uint32_t keys[];            // [slice]
  __shared__ uint32_t whist[TOPK_WARPS][256];
  __shared__ uint32_t merged[3][256];                         // cluster histogram (used in rank 0)
  __shared__ uint32_t hsum[256];                              // this pass's histogram over the row
  __shared__ int sh_scan[TOPK_WARPS + 1];
  __shared__ int sh_cnt[2];                                   // this CTA's (#greater, #ties)
  __shared__ uint32_t sh_sel[2];                              // selected digit, remaining k

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = CL > 1 ? (int)cluster.block_rank() : 0;
  const int row = blockIdx.x / CL;                            // b * Tq + i
  const int i = row % a.Tq;
  const long long t = query_pos(a.q_pos, row, i);
  int vis = t < 0 ? 0 : (int)min((long long)a.N, (t + 1) / a.m);
  if (t < 0 && rank == 0 && threadIdx.x == 0) csa_flag_error(ERRBIT_BAD_INDEX);
  const float* srow = a.scores + (size_t)row * a.N;
  int32_t* orow = a.idx + (size_t)row * a.k;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

  if (vis <= a.k) {                                           // everything visible is selected
    for (int j = rank * TOPK_THREADS + tid; j < a.k; j += CL * TOPK_THREADS)
      orow[j] = j < vis ? j : -1;
    return;
  }

  const int lo = min(vis, rank * a.slice);
  const int hi = min(vis, lo + a.slice);
  const int n = hi - lo;
  // load this CTA's slice as ordered keys (16-byte loads where aligned)
  if ((lo & 3) == 0 && ((reinterpret_cast<uintptr_t>(srow) & 15) == 0)) {
    const int n4 = n >> 2;
    const float4* s4 = reinterpret_cast<const float4*>(srow + lo);
    for (int j = tid; j < n4; j += TOPK_THREADS) {
      float4 v = __ldg(s4 + j);
      keys[4 * j] = float_to_key(v.x); keys[4 * j + 1] = float_to_key(v.y);
      keys[4 * j + 2] = float_to_key(v.z); keys[4 * j + 3] = float_to_key(v.w);
    }
    for (int j = 4 * n4 + tid; j < n; j += TOPK_THREADS) keys[j] = float_to_key(__ldg(srow + lo + j));
  } else {
    for (int j = tid; j < n; j += TOPK_THREADS) keys[j] = float_to_key(__ldg(srow + lo + j));
  }

  uint32_t prefix = 0;          // selected high digits so far
  uint32_t krem = (uint32_t)a.k;
  if constexpr (CL > 1) {
    // rank 0 collects the cluster histogram; buffer (pass % 3) is written in
    // that pass, (pass + 1) % 3 is cleared for the next one
    if (rank == 0)
      for (int j = tid; j < 2 * 256; j += TOPK_THREADS) (&merged[0][0])[j] = 0;
    cluster.sync();
  }
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const uint32_t hmask = pass == 0 ? 0u : (0xffffffffu << (shift + 8));
    for (int j = tid; j < TOPK_WARPS * 256; j += TOPK_THREADS) (&whist[0][0])[j] = 0;
    __syncthreads();
    for (int j0 = 0; j0 < n; j0 += TOPK_THREADS) {
      const int j = j0 + tid;
      bool act = false;
      uint32_t dig = 0;
      if (j < n) {
        uint32_t key = keys[j];
        act = (key & hmask) == prefix;
        dig = (key >> shift) & 255u;
      }
      uint32_t am = __ballot_sync(0xffffffffu, act);
      if (act) {
        uint32_t peers = __match_any_sync(am, dig);
        if (lane == __ffs(peers) - 1) atomicAdd(&whist[wid][dig], (uint32_t)__popc(peers));
      }
    }
    __syncthreads();
    if constexpr (CL > 1) {
      uint32_t* mrg = cluster.map_shared_rank(&merged[pass % 3][0], 0);
      for (int bin = tid; bin < 256; bin += TOPK_THREADS) {
        uint32_t s = 0;
#pragma unroll 4
        for (int w = 0; w < TOPK_WARPS; ++w) s += whist[w][bin];
        if (s) atomicAdd(mrg + bin, s);
      }
      if (rank == 0)
        for (int bin = tid; bin < 256; bin += TOPK_THREADS) merged[(pass + 1) % 3][bin] = 0;
      cluster.sync();
      for (int bin = tid; bin < 256; bin += TOPK_THREADS) hsum[bin] = mrg[bin];
    } else {
      for (int bin = tid; bin < 256; bin += TOPK_THREADS) {
        uint32_t s = 0;
#pragma unroll 4
        for (int w = 0; w < TOPK_WARPS; ++w) s += whist[w][bin];
        hsum[bin] = s;
      }
    }
    __syncthreads();
    if (wid == 0) {
      // lane l owns bins 8l..8l+7
      uint32_t cnt[8];
      uint32_t part = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        cnt[e] = hsum[8 * lane + e];
        part += cnt[e];
      }
      // suffix sums from the top lane down
      uint32_t suf = part;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += y;
      }
      const uint32_t above = suf - part;                      // count in higher lanes
      const bool here = above < krem && suf >= krem;
      if (here) {
        uint32_t run = above;
        int sel = 0;
        for (int e = 7; e >= 0; --e) {
          if (run + cnt[e] >= krem) { sel = 8 * lane + e; break; }
          run += cnt[e];
        }
        sh_sel[0] = (uint32_t)sel;
        sh_sel[1] = krem - run;
      }
    }
    __syncthreads();
    prefix |= sh_sel[0] << shift;
    krem = sh_sel[1];
  }
  // prefix = exact k-th largest key; krem = how many keys == prefix to take
  const uint32_t kth = prefix;
  int gt = 0, eq = 0;
  for (int j = tid; j < n; j += TOPK_THREADS) {
    uint32_t key = keys[j];
    gt += key > kth;
    eq += key == kth;
  }
  // CTA totals
  int tot_gt, tot_eq;
  block_excl_scan(gt, sh_scan, &tot_gt);
  block_excl_scan(eq, sh_scan, &tot_eq);
  if (tid == 0) { sh_cnt[0] = tot_gt; sh_cnt[1] = tot_eq; }
  int base_gt = 0, base_eq = 0;
  if constexpr (CL > 1) {
    cluster.sync();
    // counts of the lower ranks (lane rr reads rank rr), summed across the warp
    int g = 0, e = 0;
    if (lane < rank) {
      const int* o = cluster.map_shared_rank(sh_cnt, lane);
      g = o[0];
      e = o[1];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, off);
      e += __shfl_xor_sync(0xffffffffu, e, off);
    }
    base_gt = g;
    base_eq = e;
  } else {
    __syncthreads();
  }
  const int need_eq = (int)krem;
  const int take_before = min(need_eq, base_eq);
  const int take_here = min(sh_cnt[1], need_eq - take_before);
  int out_pos = base_gt + take_before;
  // ordered compaction: chunks of TOPK_THREADS elements, ascending index
  int eq_seen = 0;
  for (int j0 = 0; j0 < n; j0 += TOPK_THREADS) {
    const int j = j0 + tid;
    uint32_t key = j < n ? keys[j] : 0u;
    const int is_eq = (j < n && key == kth) ? 1 : 0;
    int eq_total;
    const int eq_rank = eq_seen + block_excl_scan(is_eq, sh_scan, &eq_total);
    const int sel = (j < n) && (key > kth || (is_eq && eq_rank < take_here));
    int sel_total;
    const int pos = block_excl_scan(sel, sh_scan, &sel_total);
    if (sel && out_pos + pos < a.k) orow[out_pos + pos] = lo + j;
    out_pos += sel_total;
    eq_seen += eq_total;
  }
  // -1 padding never happens here (vis > k fills all k slots)
  if constexpr (CL > 1) cluster.sync();   // keep shared memory alive for remote readers
}

}  // namespace csa
