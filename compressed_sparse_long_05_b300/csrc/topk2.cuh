// Per-row top-k by exact radix selection with candidate filtering
// (DeepSeek-V4 report, Chinese translation blog.uika.cn, §2.3.1 "top-k
// selector"; paper notes awesome.papernotes.org, C_t = TopK_k(I_t,:)).
//
// A row's visible scores [0, vis) are split over CL CTAs (a thread-block
// cluster when CL > 1), each holding its slice in shared memory as
// order-preserving uint32 keys.  Every warp owns a contiguous segment of the
// slice, so all sweeps read shared memory conflict-free and keep index order.
//
//  1. Load + 12-bit histogram of the key's top bits (warp-aggregated shared
//     atomics; merged across the cluster with DSMEM atomics into rank 0).
//  2. The threshold bin b1 holds the k-th largest key: keys above it are
//     selected outright, krem = k - #(keys above b1) remain.
//  3. Keys in b1 are copied to a candidate list (if it fits; otherwise the
//     remaining passes filter the whole slice by the b1 prefix).
//  4. Radix passes of 7 bits (the last one narrower) over the candidates find
//     the exact k-th largest key T and the number of keys equal to T to take:
//     three for float32 scores, one for bf16 scores (their keys have 16 bits,
//     so only 16 - BITS1 remain below the first digit).
//  5. Two ballot sweeps write every key > T and the lowest-index keys == T in
//     ascending index order: warp totals -> one block scan -> cluster prefix.
// Ties are broken toward the lower entry index.
#pragma once
#include <cooperative_groups.h>
#include "common.cuh"

namespace csa {
namespace cg2 = cooperative_groups;

constexpr int TK2_BITS1 = 12;                 // first digit when the kernel builds its histogram
constexpr int TK2_MAXBINS = 1 << TK2_BITS1;

struct Topk2Args {
  const void* scores;     // [rows][N] float32, or bf16 for the KEYLO = 16 kernels
  int32_t* idx;
  const int32_t* q_pos;   // [rows] query positions (null: t = i)
  int Tq, N, k, m;
  int slice;      // keys per CTA (multiple of 4)
  int cand_cap;   // candidate capacity per CTA
  uint32_t* hist;         // optional [rows][2^BITS1] first-digit histograms of the visible scores;
                          // each row's is cleared once read (left zero for the next call)
};

// dynamic shared memory: keys[slice] | cand[cand_cap] | hist1[2^BITS1] | merged1[2^BITS1]
// (merged1 only when a cluster builds the histogram itself)
__host__ __device__ constexpr size_t topk2_smem_bytes(int slice, int cand_cap, int bits1, bool merge) {
  return (size_t)slice * 4 + (size_t)cand_cap * 4 + ((size_t)4 << bits1) * (merge ? 2 : 1);
}

// Exclusive prefix over the block of one int per thread (NT threads); returns
// the total through *total.  Two __syncthreads.
template <int NT>
CSA_DEVINL int tk2_block_scan(int x, int* sh, int* total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int w = lane < NW ? sh[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < NW) sh[lane] = wi - w;
    if (lane == NW - 1) sh[NW] = wi;
  }
  __syncthreads();
  const int r = sh[wid] + incl - x;
  *total = sh[NW];
  return r;
}

// KEYLO: the lowest key bit the scores carry (0: float32 scores; 16: bf16
// scores, read as the upper half of a float32 whose lower half is zero).
template <int NT, int CL, int BITS1, int KEYLO = 0>
__global__ void __launch_bounds__(NT) topk2_kernel(const Topk2Args a) {
  if (threadIdx.x == 0) { CSA_TRACE_WALL(48); CSA_TRACE_MARK(49); }
  pdl_enter();
  constexpr int NW = NT / 32;
  constexpr int BINS1 = 1 << BITS1;
  constexpr int SHIFT1 = 32 - BITS1;
  const bool hist_in = a.hist != nullptr;
  extern __shared__ __align__(16) uint32_t tk_smem[];
  __shared__ uint32_t hist2[3][128];          // candidate-pass histograms (rank 0 merges)
  __shared__ int sh_scan[NW + 1];
  __shared__ int w_gt[NW], w_eq[NW];          // per-warp totals, then exclusive offsets
  __shared__ int sh_tot[2];                   // this CTA's (#gt, #eq), read by higher ranks
  __shared__ uint32_t sh_sel[4];              // b1 / digit, krem, cand count, T
  __shared__ int sh_cand_n;

  cg2::cluster_group cluster = cg2::this_cluster();
  const int rank = CL > 1 ? (int)cluster.block_rank() : 0;
  const int row = blockIdx.x / CL;
  const int i = row % a.Tq;
  const long long t = query_pos(a.q_pos, row, i);
  int vis = t < 0 ? 0 : (int)min((long long)a.N, (t + 1) / a.m);
  if (t < 0 && rank == 0 && threadIdx.x == 0) csa_flag_error(ERRBIT_BAD_INDEX);
  const float* srow = reinterpret_cast<const float*>(a.scores) + (size_t)row * a.N;   // KEYLO = 0
  const uint16_t* hrow = reinterpret_cast<const uint16_t*>(a.scores) + (size_t)row * a.N;   // KEYLO = 16
  int32_t* orow = a.idx + (size_t)row * a.k;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;

  if (vis <= a.k) {                                   // every visible entry is selected
    for (int j = rank * NT + tid; j < a.k; j += CL * NT) orow[j] = j < vis ? j : -1;
    if (hist_in)                                      // leave the histogram zero for the next call
      for (int j = rank * NT + tid; j < BINS1; j += CL * NT) a.hist[(size_t)row * BINS1 + j] = 0u;
    return;
  }

  uint32_t* keys = tk_smem;
  uint32_t* cand = keys + a.slice;
  uint32_t* hist1 = cand + a.cand_cap;
  uint32_t* merged1 = hist1 + BINS1;                   // cluster-built histograms only (rank 0 merges)

  const int lo = min(vis, rank * a.slice);
  const int hi = min(vis, lo + a.slice);
  const int n = hi - lo;
  // warp segments: contiguous runs of whole 32-key steps
  const int seg = (((n + NW - 1) / NW) + 31) & ~31;
  const int s0 = min(n, wid * seg), s1 = min(n, s0 + seg);

  if (hist_in) {
    const uint32_t* gh = a.hist + (size_t)row * BINS1;
    for (int j = tid; j < BINS1; j += NT) hist1[j] = gh[j];
  } else {
    for (int j = tid; j < BINS1; j += NT) hist1[j] = 0;
    if (CL > 1 && rank == 0)
      for (int j = tid; j < BINS1; j += NT) merged1[j] = 0;
  }
  if (tid < 3 * 128) (&hist2[0][0])[tid] = 0;
  if (tid == 0) {
    sh_cand_n = 0;
    sh_sel[0] = 0xffffffffu;                          // no threshold bin found (yet)
    sh_sel[1] = 0u;
  }
  if constexpr (CL > 1) cluster.sync();
  else __syncthreads();
  if (hist_in) {
    // every rank holds its copy: clear this rank's share of the row's histogram
    // so that the workspace is zero again for the next call
    uint32_t* gh = a.hist + (size_t)row * BINS1;
    for (int j = rank * (BINS1 / CL) + tid; j < (rank + 1) * (BINS1 / CL); j += NT) gh[j] = 0u;
  }

  if (tid == 0) CSA_TRACE_MARK(50);
  // ---- 1. load the slice (every copy in flight at once), then keys + first-digit histogram ----
  {
    if constexpr (KEYLO == 0) {
      const bool vec = ((lo & 3) == 0) && ((reinterpret_cast<uintptr_t>(srow) & 15) == 0);
      const int n4 = vec ? (n >> 2) : 0;
      const uint32_t kbase = (uint32_t)__cvta_generic_to_shared(keys);
      for (int j = tid; j < n4; j += NT)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(kbase + 16u * j),
                     "l"(srow + lo + 4 * j) : "memory");
      for (int j = 4 * n4 + tid; j < n; j += NT)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(kbase + 4u * j),
                     "l"(srow + lo + j) : "memory");
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    } else {
      // bf16 scores: 8 per 16-byte load, widened to the float32 bit pattern
      const bool vec = ((lo & 7) == 0) && ((reinterpret_cast<uintptr_t>(hrow) & 15) == 0);
      const int n8 = vec ? (n >> 3) : 0;
      for (int j = tid; j < n8; j += NT) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(hrow + lo) + j);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          keys[8 * j + 2 * e] = w[e] << 16;
          keys[8 * j + 2 * e + 1] = w[e] & 0xffff0000u;
        }
      }
      for (int j = 8 * n8 + tid; j < n; j += NT) keys[j] = (uint32_t)__ldg(hrow + lo + j) << 16;
    }
    __syncthreads();
    for (int j0 = s0; j0 < s1; j0 += 32) {
      const int j = j0 + lane;
      const bool act = j < s1;
      uint32_t key = 0u;
      if (act) {
        key = float_to_key(__uint_as_float(keys[j]));
        if constexpr (KEYLO == 16) key &= 0xffff0000u;   // a negative score's flip fills the low half
        keys[j] = key;
      }
      if (hist_in) continue;                          // the index kernel built the histogram
      const uint32_t am = __ballot_sync(0xffffffffu, act);
      if (act) {
        const uint32_t dig = key >> SHIFT1;
        const uint32_t peers = __match_any_sync(am, dig);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist1[dig], (uint32_t)__popc(peers));
      }
    }
  }
  __syncthreads();
  if (CL > 1 && !hist_in) {
    uint32_t* dst = cluster.map_shared_rank(merged1, 0);
    for (int b = tid; b < BINS1; b += NT) {
      const uint32_t c = hist1[b];
      if (c) atomicAdd(dst + b, c);
    }
    cluster.sync();
    for (int b = tid; b < BINS1; b += NT) hist1[b] = dst[b];
    __syncthreads();
  }

  // ---- 2. threshold bin: suffix counts over the first digit ----
  {
    constexpr int PER = BINS1 / NT;                   // bins per thread (>= 2)
    const int rt = NT - 1 - tid;                      // thread rt holds the highest bins first
    uint32_t c[PER];
    int part = 0;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      c[e] = hist1[rt * PER + e];
      part += (int)c[e];
    }
    int tot;
    const int above = tk2_block_scan<NT>(part, sh_scan, &tot);   // keys in bins above this thread's
    if (tot != vis) {
      // the histogram does not count exactly the row's visible keys (a stale or
      // partial caller-side histogram): no threshold is taken from it
      if (tid == 0) sh_sel[0] = 0xfffffffeu;
    } else if (above < a.k && above + part >= a.k) {
      int run = above;
#pragma unroll
      for (int e = PER - 1; e >= 0; --e) {
        if (run + (int)c[e] >= a.k) {
          sh_sel[0] = (uint32_t)(rt * PER + e);
          sh_sel[1] = (uint32_t)(a.k - run);
          sh_sel[2] = c[e];
          break;
        }
        run += (int)c[e];
      }
    }
    __syncthreads();
  }
  if (sh_sel[0] >= 0xfffffffeu) {
    // the histogram does not describe these scores (its total is not the
    // visible count, or it holds fewer than k keys; only a broken caller-side
    // histogram gets here).  Flag it and leave the row empty rather than
    // select from a wrong threshold.
    if (tid == 0 && rank == 0) csa_flag_error(ERRBIT_HIST);
    for (int j = rank * NT + tid; j < a.k; j += CL * NT) orow[j] = -1;
    if constexpr (CL > 1) cluster.sync();             // no rank leaves while peers may map its memory
    return;
  }
  const uint32_t b1 = sh_sel[0];
  uint32_t krem = sh_sel[1];
  if (tid == 0) CSA_TRACE_MARK(51);

  // ---- 3. candidates: this slice's keys in bin b1 ----
  int ncand = 0;
  bool cand_ok;
  {
    // count this slice's b1 keys first (capacity check), then copy
    int mine = 0;
    for (int j = s0 + lane; j < s1; j += 32) mine += (keys[j] >> SHIFT1) == b1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
    if (lane == 0) atomicAdd(&sh_cand_n, mine);
    __syncthreads();
    ncand = sh_cand_n;
    cand_ok = ncand <= a.cand_cap;
    __syncthreads();
    if (cand_ok) {
      if (tid == 0) sh_cand_n = 0;
      __syncthreads();
      for (int j0 = s0; j0 < s1; j0 += 32) {
        const int j = j0 + lane;
        const uint32_t key = j < s1 ? keys[j] : 0u;
        const bool in = j < s1 && (key >> SHIFT1) == b1;
        const uint32_t bm = __ballot_sync(0xffffffffu, in);
        if (bm) {
          int base = 0;
          if (lane == 0) base = atomicAdd(&sh_cand_n, __popc(bm));
          base = __shfl_sync(0xffffffffu, base, 0);
          if (in) cand[base + __popc(bm & lt_mask)] = key;
        }
      }
      __syncthreads();
    }
  }
  const uint32_t* list = cand_ok ? cand : keys;
  const int list_n = cand_ok ? ncand : n;
  if (tid == 0) CSA_TRACE_MARK(52);

  // ---- 4. three radix passes over the candidates (or the b1-filtered slice) ----
  uint32_t prefix = b1 << SHIFT1;
  uint32_t pmask = 0xffffffffu << SHIFT1;
  // the bits [KEYLO, SHIFT1) below the first digit, 7 at a time from the top
  constexpr int NPASS = (SHIFT1 - KEYLO + 6) / 7;
#pragma unroll 1
  for (int pass = 0; pass < NPASS; ++pass) {
    const int hi_bit = SHIFT1 - 7 * pass;
    const int wd = hi_bit - KEYLO < 7 ? hi_bit - KEYLO : 7;
    const int sh = hi_bit - wd;
    const uint32_t dmask = (1u << wd) - 1u;
    uint32_t* h = hist2[pass];
    for (int j0 = 0; j0 < list_n; j0 += NT) {
      const int j = j0 + tid;
      bool act = false;
      uint32_t dig = 0;
      if (j < list_n) {
        const uint32_t key = list[j];
        act = (key & pmask) == prefix;
        dig = (key >> sh) & dmask;
      }
      const uint32_t am = __ballot_sync(0xffffffffu, act);
      if (act) {
        const uint32_t peers = __match_any_sync(am, dig);
        if (lane == __ffs(peers) - 1) atomicAdd(&h[dig], (uint32_t)__popc(peers));
      }
    }
    __syncthreads();
    if constexpr (CL > 1) {
      uint32_t* dst = cluster.map_shared_rank(&hist2[pass][0], 0);
      if (rank != 0 && tid < 128) {
        const uint32_t c = h[tid];
        if (c) atomicAdd(dst + tid, c);
      }
      cluster.sync();
      if (tid < 128) h[tid] = dst[tid];
      __syncthreads();
    }
    if (wid == 0) {
      // every thread's reads of the previous pass's selection ended at the
      // barrier above: mark "no digit found" before this pass selects
      if (lane == 0) sh_sel[0] = 0xffffffffu;
      __syncwarp();
      // lane l holds digits 4l..4l+3 (128 bins; unused high bins are zero)
      uint32_t c[4];
      uint32_t part = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) { c[e] = h[4 * lane + e]; part += c[e]; }
      uint32_t suf = part;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += y;
      }
      const uint32_t above = suf - part;
      if (above < krem && suf >= krem) {
        uint32_t run = above;
#pragma unroll
        for (int e = 3; e >= 0; --e) {
          if (run + c[e] >= krem) { sh_sel[0] = (uint32_t)(4 * lane + e); sh_sel[1] = krem - run; break; }
          run += c[e];
        }
      }
    }
    __syncthreads();
    if (sh_sel[0] == 0xffffffffu) {
      // fewer candidates than the histogram promised: same treatment as above
      // (every rank merged the same counts, so the whole cluster leaves here)
      if (tid == 0 && rank == 0) csa_flag_error(ERRBIT_HIST);
      for (int j = rank * NT + tid; j < a.k; j += CL * NT) orow[j] = -1;
      if constexpr (CL > 1) cluster.sync();
      return;
    }
    prefix |= sh_sel[0] << sh;
    pmask |= dmask << sh;
    krem = sh_sel[1];
  }
  if (tid == 0) CSA_TRACE_MARK(53);
  const uint32_t T = prefix;          // exact k-th largest key
  const int q_eq = (int)krem;         // keys == T to take, lowest indices first

  // ---- 5. ordered output ----
  int g_w = 0, e_w = 0;
  for (int j0 = s0; j0 < s1; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t key = j < s1 ? keys[j] : 0u;
    g_w += __popc(__ballot_sync(0xffffffffu, j < s1 && key > T));
    e_w += __popc(__ballot_sync(0xffffffffu, j < s1 && key == T));
  }
  if (lane == 0) { w_gt[wid] = g_w; w_eq[wid] = e_w; }
  __syncthreads();
  if (wid == 0) {
    int g = lane < NW ? w_gt[lane] : 0, e = lane < NW ? w_eq[lane] : 0;
    int gi = g, ei = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y1 = __shfl_up_sync(0xffffffffu, gi, o);
      const int y2 = __shfl_up_sync(0xffffffffu, ei, o);
      if (lane >= o) { gi += y1; ei += y2; }
    }
    if (lane < NW) { w_gt[lane] = gi - g; w_eq[lane] = ei - e; }
    if (lane == NW - 1) { sh_tot[0] = gi; sh_tot[1] = ei; }
  }
  int base_gt = 0, base_eq = 0;
  if constexpr (CL > 1) {
    cluster.sync();
    int g = 0, e = 0;
    if (lane < rank) {
      const int* o = cluster.map_shared_rank(sh_tot, lane);
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
  int gt_before = base_gt + w_gt[wid];
  int eq_before = base_eq + w_eq[wid];
  for (int j0 = s0; j0 < s1; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t key = j < s1 ? keys[j] : 0u;
    const uint32_t gm = __ballot_sync(0xffffffffu, j < s1 && key > T);
    const uint32_t em = __ballot_sync(0xffffffffu, j < s1 && key == T);
    const int g_lt = gt_before + __popc(gm & lt_mask);
    const int e_lt = eq_before + __popc(em & lt_mask);
    const bool take = j < s1 && (key > T || (key == T && e_lt < q_eq));
    if (take) {
      const int pos = g_lt + min(q_eq, e_lt);
      if (pos >= 0 && pos < a.k) orow[pos] = lo + j;
    }
    gt_before += __popc(gm);
    eq_before += __popc(em);
  }
  if (tid == 0) CSA_TRACE_MARK(54);
  if constexpr (CL > 1) cluster.sync();   // peers may still read sh_tot / histograms
  if (tid == 0) { CSA_TRACE_MARK(56); CSA_TRACE_WALL(55); }
}

}  // namespace csa
