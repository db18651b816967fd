// Shared-KV multi-query core attention on the tcgen05 tensor cores
// (d = 512, RoPE on the last 64 dims, bf16 rows and queries).
//
// DeepSeek-V4 report (Chinese translation, blog.uika.cn) §2.3.1 "Shared KV
// MQA" (each selected compressed entry is both key and value, all query heads
// share it), §2.3.2 (HCA: every visible compressed entry), §2.3.3 (partial
// RoPE with the output rotated back at -t, 128-token sliding window, per-head
// attention sink in the softmax denominator).
//
// One CTA handles one work item = (query row, group of 64 heads, chunk of the
// row set).  The row set of query t is its selected compressed entries (or,
// for HCA, every visible one) followed by the raw window tokens; rows are
// gathered 128 at a time into shared memory as a 128-byte-swizzled tile E
// [128 rows x 512 dims].  The same bytes are the K-major A operand of
//     S^T[128 rows x 64 heads]  = E * Q^T            (tcgen05, M=128, N=64, K=512)
// and the MN-major A operand of
//     O^T[512 dims x 64 heads] += E^T * P^T          (4 MMAs of M=128, N=64, K=128)
// so one tile feeds both products without a transpose.  O^T (4 x 64 columns)
// and two S^T buffers (2 x 64) live in tensor memory.
//
// Softmax runs over rows (TMEM lanes) per head (column): each warp reduces its
// 32 rows with a reduce-scatter butterfly (lane l ends with heads 2l, 2l+1),
// warps combine through shared memory behind mbarriers.  The running max is
// raised lazily (only when a tile's max exceeds it by 8 in log2 units), so O^T
// is rescaled in tensor memory only on those rare tiles.  P^T is written as
// bf16 and the row sums use the same rounded values.
//
// Warp roles (288 threads): warps 0-3 softmax / epilogue (one TMEM lane
// quarter each), warps 4-7 gather (32 rows each), warp 8 TMEM owner + MMA
// issuer.
//   - bf16 rows are copied with cp.async, 16 bytes per lane straight into the
//     swizzled tile; each lane's copies of a 64-dim chunk arrive on that
//     chunk's barrier as they land (measured faster than TMA tile::gather4,
//     which this tile layout also allows).
//   - FP8 / BF16-RoPE rows are copied with cp.async (all of a tile at once)
//     and widened to bf16 in place.
//   - RoPE: when many query rows share few stored rows (prefill), every stored
//     row is rotated once up front at its absolute position and the query is
//     rotated at t (output rotated back at -t).  Otherwise (decode) each
//     gathered row is rotated in shared memory by (position - t), so the query
//     (loaded unrotated by TMA) and the output need no rotation.
//   - The first tile of an item fetches each row's 1 KB together; later tiles
//     refill each chunk pair as soon as the PV block that read it is done.
//
// A single-chunk item finishes in the kernel: divide by the softmax
// denominator plus exp(sink), rotate the RoPE dims back if needed, store bf16.
// A multi-chunk item (decode: few query rows, many rows each) keeps its
// unnormalised O and its running max and denominator, and the chunks merge by
// log-sum-exp, in one of two ways:
//   - cluster merge: the chunks of a (query row, head group) run as one thread-
//     block cluster, each staging its O (fp32 [64 heads][512 dims]) and (max,
//     sum) in its own shared memory; every CTA then merges its share of the
//     outputs from all chunks' shared memory over DSMEM and stores bf16;
//   - otherwise O goes to global memory (one bulk copy of the staged tile when
//     the CTA has one item) and attend_combine_kernel merges.
#pragma once
#include <cooperative_groups.h>
#include <cuda_fp8.h>
#include "tc.cuh"

namespace csa {

constexpr int ATT_THREADS = 288;
constexpr int ATT_D = 512;
constexpr int ATT_R = 64;
constexpr int ATT_HG = 64;          // heads per CTA
constexpr int ATT_TILE = 128;       // rows per tile
constexpr float ATT_TAU = 8.0f;     // lazy-rescale threshold (log2 units)

struct AttendTcArgs {
  const __nv_bfloat16* q;        // [B, Tq, n_h, 512]
  const void* ent;               // [B, N, 512] bf16 (or e4m3 nope, see kv_mixed)
  const float* ent_scale;        // [B, N] (kv_mixed)
  const __nv_bfloat16* ent_rope; // [B, N, 64] (kv_mixed)
  const void* win;               // [B, T_win, 512] bf16 (or e4m3 nope)
  const float* win_scale;
  const __nv_bfloat16* win_rope;
  const int32_t* idx;            // [B, Tq, k] or null (dense)
  const int32_t* q_pos;          // [B, Tq] query positions (null: t = i)
  const int32_t* win_base;       // [B] token of window row 0 (null: 0)
  const float* sink;             // [n_h]
  __nv_bfloat16* out;            // [B, Tq, n_h, 512]
  float* part_o;                 // [items][64 heads][512 dims] (split mode)
  float* part_ml;                // [items][64][2]   (split mode)
  int B, Tq, N, k, T_win, n_h, m, n_win;
  int HG;                        // head groups = n_h / 64
  int nch;                       // chunks per (query row, head group)
  int chunk_rows;                // rows per chunk (multiple of 128)
  int items;                     // B * Tq * HG * nch
  int rotate_rows;               // 1 = rotate gathered rows in shared memory
  int rel_rope;                  // 1 = rows rotated by (position - t): q and out stay unrotated
  int kv_mixed;                  // 1 = e4m3 + scale + bf16 rope rows
  int cl_reduce;                 // 1 = clusters of ncs consecutive chunks merge over DSMEM
  int ncs;                       // chunks per cluster (cl_reduce): nch, or a divisor of it
  int cl_partial;                // 1 = each cluster merges its ncs chunks into one fp32 partial
                                 //     (part_o / part_ml at index item / ncs) for the combine kernel
  int ent_rotated;               // 1 = entries stored with their RoPE dims already rotated at m(s+1)-1
  RowPages ent_pg, win_pg;       // paged / ring row maps (no table: flat)
  float scale_log2;              // log2(e) / sqrt(d)
  RopeFreqs rf;
};

struct AttSmem {
  static constexpr int E = 0;                              // 8 chunks x 16 KB
  static constexpr int Q = E + 8 * 16384;                  // 8 chunks x 8 KB
  static constexpr int P = Q + 8 * 8192;                   // 128 rows x 128 B
  static constexpr int MAXP = P + 16384;                   // [2][4][64] f32
  static constexpr int SUMP = MAXP + 2 * 4 * 64 * 4;       // [2][4][64] f32
  static constexpr int MROW = SUMP + 2 * 4 * 64 * 4;       // [4 warps][64] f32 running max
  static constexpr int FAC = MROW + 4 * 64 * 4;            // [4][64] f32 rescale factors
  static constexpr int ML = FAC + 4 * 64 * 4;              // [64][2] f32 this chunk's (max, sum) (cluster merge)
  static constexpr int MLALL = ML + 64 * 2 * 4;            // [16 chunks][64][2] f32 every chunk's (max, sum)
  static constexpr int OWNW = MLALL + 16 * 64 * 2 * 4;     // [64] f32 this chunk's merge weight
  static constexpr int INVD = OWNW + 64 * 4;               // [64] f32 1 / denominator (cluster merge)
  static constexpr int SINK = INVD + 64 * 4;               // [64] f32 sink logits of the head group, in log2 units
  static constexpr int RMASK = SINK + 64 * 4;              // [2 tiles][4 warps] u32 row-valid bits
  static constexpr int ROPEF = RMASK + 64;                 // [64] u64 RoPE phase steps (copy of the args)
  static constexpr int BAR = ROPEF + 64 * 8;
  static constexpr int NBAR = 32;
  static constexpr int MISC = BAR + NBAR * 8;
  static constexpr int BYTES = MISC + 64 + 1024;           // + alignment slack
};

// row set of one query row
struct AttRow {
  int b, i, hg, c;
  long long t;
  int nsel;        // compressed rows (selected or visible)
  long long w0;    // first window token
  long long wbase; // token of window buffer row 0 of batch row b
  int nrows;       // nsel + window size
  int r0, r1;      // this chunk's rows [r0, r1)
};

// The row set of work item `it`.  A negative position has no rows (its output
// is zero); the gather warps flag it.
CSA_DEVINL AttRow att_item(const AttendTcArgs& a, int it) {
  AttRow x;
  x.c = it % a.nch;
  int rest = it / a.nch;
  x.hg = rest % a.HG;
  rest /= a.HG;
  x.i = rest % a.Tq;
  x.b = rest / a.Tq;
  x.t = query_pos(a.q_pos, (long long)x.b * a.Tq + x.i, x.i);
  x.wbase = window_base(a.win_base, x.b);
  if (x.t < 0) {
    x.nsel = 0;
    x.w0 = 0;
    x.nrows = 0;
  } else {
    long long vis = (x.t + 1) / a.m;
    if (vis > a.N) vis = a.N;
    x.nsel = a.idx ? (int)min((long long)a.k, vis) : (int)vis;
    x.w0 = x.t - a.n_win + 1;
    if (x.w0 < 0) x.w0 = 0;
    x.nrows = x.nsel + (int)(x.t - x.w0 + 1);
  }
  x.r0 = min(x.nrows, x.c * a.chunk_rows);
  x.r1 = min(x.nrows, x.r0 + a.chunk_rows);
  return x;
}

CSA_DEVINL void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
CSA_DEVINL void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 32 lanes x 8 consecutive 32-bit columns (load and store)
CSA_DEVINL void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
CSA_DEVINL void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

CSA_DEVINL void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
CSA_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Arrive on `bar` once every cp.async this thread issued so far has landed (the
// barrier's pending count is raised by one until then).
CSA_DEVINL void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
template <int N>
CSA_DEVINL void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// rotate the 4 (x0, x1) pairs of one 16-byte bf16 unit; pair p uses frequency j0 + p.
// F is the CTA's shared-memory copy of the phase steps: lanes read different
// frequencies, which a kernel-parameter array would serve one address at a time.
CSA_DEVINL uint4 rope_unit(uint4 v, long long pos, const unsigned long long* F, int j0) {
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w[p]);
    float2 f = __bfloat1622float2(h);
    float c, s;
    rope_cos_sin(pos, F[j0 + p], c, s);
    w[p] = pack_bf16x2(f.x * c - f.y * s, f.x * s + f.y * c);
  }
  return v;
}

// 2^x on the special-function unit (one instruction; flushes results below
// 2^-126 to zero, which a softmax weight can take)
CSA_DEVINL float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// reduce-scatter butterfly over the warp of 64 values per lane, read through
// get(e) (so the caller's values need not be copied): on exit lane l holds in
// r[0], r[1] the op-reduced columns 2l and 2l+1 over all 32 lanes.
template <bool IS_MAX, typename Get>
CSA_DEVINL void warp_reduce_scatter64_from(Get get, float* r, int lane) {
  {
    const bool upper = (lane & 16) != 0;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float lo = get(e), hi = get(e + 32);
      const float send = upper ? lo : hi;
      const float keep = upper ? hi : lo;
      const float got = __shfl_xor_sync(0xffffffffu, send, 16);
      r[e] = IS_MAX ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int lvl = 1; lvl < 5; ++lvl) {
    const int off = 16 >> lvl;        // partner distance
    const int hs = 32 >> lvl;         // half of the values still held
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int e = 0; e < hs; ++e) {
      const float lo = r[e], hi = r[e + hs];
      const float send = upper ? lo : hi;
      const float keep = upper ? hi : lo;
      const float got = __shfl_xor_sync(0xffffffffu, send, off);
      r[e] = IS_MAX ? fmaxf(keep, got) : keep + got;
    }
  }
}

// reduce-scatter butterfly over the warp: on entry x[0..63] per lane; on exit
// lane l holds op-reduced columns 2l (x[0]) and 2l+1 (x[1]) over all 32 lanes.
template <bool IS_MAX>
CSA_DEVINL void warp_reduce_scatter64(float* x, int lane) {
#pragma unroll
  for (int lvl = 0; lvl < 5; ++lvl) {
    const int off = 16 >> lvl;        // partner distance
    const int hs = 32 >> lvl;         // half of the values still held
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int e = 0; e < hs; ++e) {
      const float lo = x[e], hi = x[e + hs];
      const float send = upper ? lo : hi;
      const float keep = upper ? hi : lo;
      const float got = __shfl_xor_sync(0xffffffffu, send, off);
      x[e] = IS_MAX ? fmaxf(keep, got) : keep + got;
    }
  }
}

// eight e4m3 bytes times the row scale -> eight bf16 (one 16-byte unit)
CSA_DEVINL uint4 e4m3x8_to_bf16(uint2 raw, float scale) {
  float f[8];
  const __nv_fp8x2_storage_t* p2 = reinterpret_cast<const __nv_fp8x2_storage_t*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(p2[e], __NV_E4M3);
    __half2 h2 = *reinterpret_cast<__half2*>(&hr);
    float2 v = __half22float2(h2);
    f[2 * e] = v.x * scale;
    f[2 * e + 1] = v.y * scale;
  }
  return f_to_bf16x8(f);
}

// Cluster merge of a head group's chunks (one item per CTA; cluster rank = chunk).
// Output dims are split among the CTAs in groups of 8: CTA o owns dim groups
// [ceil(64 o / nch), ceil(64 (o+1) / nch)).
//  1. every CTA sends its per-head (max, sum) into every peer's MLALL slot
//     (st.async, completing on the peer's ml_bar); a CTA sends only after its
//     own PV is done, so once a CTA holds everyone's values, every CTA's E / Q
//     region is free to receive partials;
//  2. meanwhile eight warps read this chunk's O^T from TMEM (one dim, 64 heads
//     per thread) and stage it as bf16 in local shared memory grouped by
//     owner ([owner][head][pitch]); a chunk that saw no row stages zeros;
//  3. once every (max, sum) is in, one DSMEM bulk copy per owner moves that
//     owner's block into its receive buffer ([chunk][head][pitch]),
//     completing on the owner's merge_bar;
//  4. while the copies fly, each CTA computes for every chunk c and head h the
//     weight 2^(m_c - M_h) / (sum_c' l_c' 2^(m_c' - M_h) + 2^(z'_h - M_h)),
//     M_h the largest of the chunks' maxima and the sink logit;
//  5. each owner waits for its nch blocks and, per head and group of 8 dims,
//     accumulates weight * partial in fp32 from 16-byte vectors and stores 8
//     bf16 outputs at once (relative-RoPE mode: no output rotation).
// Every CTA waits for each byte destined to it before it leaves, so no cluster
// barrier is needed after the copies.  The partials are rounded to bf16 once
// (relative 2^-9) before the fp32 sum.
CSA_DEVINL int merge_dim_lo(int o, int nch) { return 8 * ((o * (ATT_D / 8) + nch - 1) / nch); }
// dims per head row of a staged / received block: the largest owner's, in 8s
CSA_DEVINL int merge_pitch(int nch) { return 8 * ((ATT_D / 8 + nch - 1) / nch); }
constexpr int MERGE_RECV = 80 * 1024;   // receive buffer offset in the E / Q region

CSA_DEVINL uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

CSA_DEVINL void st_async_f2(uint32_t addr, float a0, float a1, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
               ::"r"(addr), "f"(a0), "f"(a1), "r"(mbar)
               : "memory");
}

CSA_DEVINL void attend_cluster_merge(const AttendTcArgs& a, uint8_t* smem, uint32_t tmem,
                                     uint64_t* merge_bar, uint64_t* ml_bar) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int nch = a.ncs;                              // chunks merged by this cluster
  const int crank = (int)cl.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttRow x = att_item(a, blockIdx.x);
  const float* ml = reinterpret_cast<const float*>(smem + AttSmem::ML);
  float* mlall = reinterpret_cast<float*>(smem + AttSmem::MLALL);     // [chunk][64][2]: (m, l), then weights
  const int pitch = merge_pitch(nch);
  const uint32_t blk = (uint32_t)(ATT_HG * pitch * 2);                 // bytes of one block
  __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem + AttSmem::E);   // [owner][64][pitch]
  __nv_bfloat16* recv = reinterpret_cast<__nv_bfloat16*>(smem + AttSmem::E + MERGE_RECV);  // [chunk][64][pitch]
  const int lo = merge_dim_lo(crank, nch), dn = merge_dim_lo(crank + 1, nch) - lo;
  volatile int no_abort = 0;   // the merge's waits end on data, never on a role's abort
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every peer has started
  for (int i = threadIdx.x; i < nch * ATT_HG; i += blockDim.x) {
    const int c = i / ATT_HG, h = i % ATT_HG;
    st_async_f2(mapa_shared(smem_u32(mlall + (crank * ATT_HG + h) * 2), (uint32_t)c), ml[2 * h],
                ml[2 * h + 1], mapa_shared(smem_u32(ml_bar), (uint32_t)c));
  }
  if (warp < 8) {
    // stage this chunk's O (needs nothing from the peers): warp w reads TMEM
    // lane quarter w % 4 (dims bk*128 + (w%4)*32 + lane) for the dim blocks
    // bk = 2 (w / 4) and 2 (w / 4) + 1
    const int q4 = warp & 3;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const bool has_o = reinterpret_cast<const int*>(smem + AttSmem::MISC)[2] != 0;
#pragma unroll 1
    for (int bb = 0; bb < 2; ++bb) {
      const int bk = 2 * (warp >> 2) + bb;
      const int dim = bk * 128 + q4 * 32 + lane;
      const int o = (dim >> 3) * nch / (ATT_D / 8);
      __nv_bfloat16* dst = stage + (size_t)o * ATT_HG * pitch + (dim - merge_dim_lo(o, nch));
      uint32_t r[64];
      if (has_o) {
        tmem_ld32(tmem + lane_base + bk * ATT_HG, r);
        tmem_ld32(tmem + lane_base + bk * ATT_HG + 32, r + 32);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int h = 0; h < 64; ++h) r[h] = 0u;      // no row: TMEM holds no O
      }
#pragma unroll
      for (int h = 0; h < ATT_HG; ++h) dst[(size_t)h * pitch] = __float2bfloat16_rn(__uint_as_float(r[h]));
    }
  }
  fence_proxy_async();                                // staged bytes -> visible to the bulk copies
  if (threadIdx.x == 0) CSA_TRACE_MARK(17);
  // every chunk's (max, sum) is here, so every peer's PV is done and its
  // receive buffer is free
  mbar_wait(ml_bar, 0, &no_abort);
  __syncthreads();
  if (threadIdx.x == 0) CSA_TRACE_MARK(18);
  if (threadIdx.x < (unsigned)nch) {
    // block of owner o -> owner's recv[crank]
    const int o = threadIdx.x;
    const uint32_t src = smem_u32(stage) + (uint32_t)o * blk;
    const uint32_t dst = mapa_shared(smem_u32(recv) + (uint32_t)crank * blk, (uint32_t)o);
    const uint32_t bar = mapa_shared(smem_u32(merge_bar), (uint32_t)o);
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "r"(src), "r"(blk), "r"(bar)
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
  // while the copies fly: the weight of every (chunk, head),
  // 2^(m_c - M_h) / (sum_c' l_c' 2^(m_c' - M_h) + 2^(z'_h - M_h)), written over m_c
  if (a.cl_partial && threadIdx.x >= 32 && threadIdx.x < 32 + ATT_HG) {
    // partial of this cluster's chunks: weights 2^(m_c - M), and (M, sum_c l_c 2^(m_c - M))
    // for the combine kernel (no sink, no normalisation here)
    const int h = threadIdx.x - 32;
    float M = -INFINITY;
    for (int k = 0; k < nch; ++k)
      if (mlall[(k * ATT_HG + h) * 2 + 1] > 0.f) M = fmaxf(M, mlall[(k * ATT_HG + h) * 2]);
    float L = 0.f;
    for (int k = 0; k < nch; ++k) {
      const float lk = mlall[(k * ATT_HG + h) * 2 + 1];
      const float ek = lk > 0.f ? exp2f(mlall[(k * ATT_HG + h) * 2] - M) : 0.f;
      mlall[(k * ATT_HG + h) * 2] = ek;
      L += lk * ek;
    }
    if (crank == 0) {
      float* pm = a.part_ml + ((size_t)(blockIdx.x / nch) * ATT_HG + h) * 2;
      pm[0] = M;
      pm[1] = L;
    }
  } else if (threadIdx.x >= 32 && threadIdx.x < 32 + ATT_HG) {
    const int h = threadIdx.x - 32;
    const float zs = reinterpret_cast<const float*>(smem + AttSmem::SINK)[h];
    float M = zs;
    for (int k = 0; k < nch; ++k)
      if (mlall[(k * ATT_HG + h) * 2 + 1] > 0.f) M = fmaxf(M, mlall[(k * ATT_HG + h) * 2]);
    float den = exp2f(zs - M);
    for (int k = 0; k < nch; ++k) {
      const float lk = mlall[(k * ATT_HG + h) * 2 + 1];
      const float ek = lk > 0.f ? exp2f(mlall[(k * ATT_HG + h) * 2] - M) : 0.f;
      mlall[(k * ATT_HG + h) * 2] = ek;
      den += lk * ek;
    }
    const float inv = 1.f / den;
    for (int k = 0; k < nch; ++k) mlall[(k * ATT_HG + h) * 2] *= inv;
  }
  __syncthreads();
  if (threadIdx.x == 0) CSA_TRACE_MARK(19);
  // this CTA's blocks from every chunk (they must land before it may leave)
  const bool got = mbar_wait(merge_bar, 0, &no_abort);
  if (threadIdx.x == 0) CSA_TRACE_MARK(20);
  if (got) {
    const size_t orow = ((size_t)x.b * a.Tq + x.i) * a.n_h + (size_t)x.hg * ATT_HG;
    const int ng = dn >> 3;                           // groups of 8 dims this CTA owns
    for (int i = threadIdx.x; i < ATT_HG * ng; i += blockDim.x) {
      const int h = i / ng, g = i - h * ng;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
      const uint4* src = reinterpret_cast<const uint4*>(recv + (size_t)h * pitch + 8 * g);
      for (int c = 0; c < nch; ++c) {
        const float w = mlall[(c * ATT_HG + h) * 2];
        float f[8];
        bf16x8_to_f(src[(size_t)c * ATT_HG * pitch / 8], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(w, f[e], acc[e]);
      }
      if (a.cl_partial) {
        float4* po = reinterpret_cast<float4*>(
            a.part_o + ((size_t)(blockIdx.x / nch) * ATT_HG + h) * ATT_D + lo + 8 * g);
        po[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        po[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      } else {
        *reinterpret_cast<uint4*>(a.out + (orow + h) * ATT_D + lo + 8 * g) = f_to_bf16x8(acc);
      }
    }
  }
  if (threadIdx.x == 0) CSA_TRACE_MARK(26);
  if (threadIdx.x < (unsigned)nch)                    // own copies have read their source
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  if (threadIdx.x == 0) CSA_TRACE_MARK(27);
}

__global__ void __launch_bounds__(ATT_THREADS, 1)
attend_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const AttendTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem<1024>(smem_raw);
  uint8_t* sE = smem + AttSmem::E;
  uint8_t* sQ = smem + AttSmem::Q;
  uint8_t* sP = smem + AttSmem::P;
  float* maxp = reinterpret_cast<float*>(smem + AttSmem::MAXP);
  float* sump = reinterpret_cast<float*>(smem + AttSmem::SUMP);
  float* mrow = reinterpret_cast<float*>(smem + AttSmem::MROW);
  float* facs = reinterpret_cast<float*>(smem + AttSmem::FAC);
  volatile uint32_t* rmask = reinterpret_cast<volatile uint32_t*>(smem + AttSmem::RMASK);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + AttSmem::BAR);
  uint64_t* chunk_full = bar;        // [8]  gather warps -> MMA (count 4)
  uint64_t* chunk_free = bar + 8;    // [4]  PV block done -> gather (commit)
  uint64_t* s_full = bar + 12;       // [2]  QK done -> softmax (commit)
  uint64_t* s_free = bar + 14;       // [2]  softmax read S -> MMA (count 4)
  uint64_t* p_full = bar + 16;       // P^T written (+ O rescaled) -> MMA (count 4)
  uint64_t* p_free = bar + 17;       // PV done (commit)
  uint64_t* q_full = bar + 18;       // Q staged -> MMA (count 4)
  uint64_t* q_free = bar + 19;       // last QK of the item done (commit)
  uint64_t* o_free = bar + 20;       // epilogue read O -> MMA (count 4)
  uint64_t* grp_a = bar + 21;        // softmax warps: tile max partials (count 4)
  uint64_t* grp_b = bar + 22;        // softmax warps: sum partials (count 4)
  uint64_t* mma_done = bar + 23;
  uint64_t* q_ready = bar + 24;      // absolute-RoPE mode: q rotated at t -> MMA (count 4)
  uint64_t* merge_bar = bar + 25;    // cluster merge: this CTA's slices from every chunk landed
  uint64_t* ml_bar = bar + 26;       // cluster merge: every chunk's (max, sum) landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + AttSmem::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + AttSmem::MISC + 4);
  unsigned long long* ropeF = reinterpret_cast<unsigned long long*>(smem + AttSmem::ROPEF);
  if (threadIdx.x < 64) ropeF[threadIdx.x] = a.rf.F[threadIdx.x];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) { CSA_TRACE_WALL(0); CSA_TRACE_MARK(1); }

  if (threadIdx.x == 0) {
    for (int c = 0; c < 8; ++c) mbar_init(chunk_full + c, 4);
    for (int c = 0; c < 4; ++c) mbar_init(chunk_free + c, 1);
    for (int s = 0; s < 2; ++s) { mbar_init(s_full + s, 1); mbar_init(s_free + s, 4); }
    mbar_init(p_full, 4);
    mbar_init(p_free, 1);
    mbar_init(q_full, 1);
    mbar_init(q_ready, 4);
    mbar_init(q_free, 1);
    mbar_init(o_free, 4);
    mbar_init(grp_a, 4);
    mbar_init(grp_b, 4);
    mbar_init(mma_done, 1);
    mbar_init(merge_bar, 1);
    mbar_init(ml_bar, 1);
    if (a.cl_reduce) {
      // the merge receives nch (max, sum) sets and nch blocks of partials
      const int pitch = merge_pitch(a.ncs);
      mbar_arrive_expect_tx(ml_bar, (uint32_t)(a.ncs * ATT_HG * 8));
      mbar_arrive_expect_tx(merge_bar, (uint32_t)(a.ncs * ATT_HG * pitch * 2));
    }
    *abort_flag = 0;
    reinterpret_cast<volatile int*>(smem + AttSmem::MISC)[2] = 0;   // this CTA's O holds rows
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // cluster merge: announce that this CTA runs (peers wait for it before their
  // first store into this CTA's shared memory)
  if (a.cl_reduce) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  // Barriers and tensor memory are set up; the previous kernel may still run
  // (programmatic launch): no global memory is read before this wait.
  pdl_enter();
  if (threadIdx.x == 0) CSA_TRACE_MARK(2);
  const uint32_t TM_O = 0, TM_S = 256;     // O^T blocks at 0..255, S^T buffers at 256..383
  if (a.cl_reduce && threadIdx.x < ATT_HG) {
    // the merge's sink logits, fetched now rather than on its critical path
    // (softmax warps 0-1 have no S to read for microseconds yet); the barrier
    // before the merge publishes them
    const int hg = (int)((blockIdx.x / a.nch) % a.HG);
    reinterpret_cast<float*>(smem + AttSmem::SINK)[threadIdx.x] =
        __ldg(a.sink + hg * ATT_HG + threadIdx.x) * 1.4426950408889634f;
  }

  if (warp >= 4 && warp < 8) {
    // ======================= gather warps =======================
    const int gw = warp - 4;
    uint32_t n = 0, nitem = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
      const AttRow x = att_item(a, it);
      if (n == 0 && gw == 0 && lane == 0) CSA_TRACE_MARK(31);
      if (x.t < 0 && gw == 0 && lane == 0 && x.c == 0 && x.hg == 0) csa_flag_error(ERRBIT_BAD_INDEX);
      if (x.r1 <= x.r0) continue;
      // ---- tiles ----
      for (int r0 = x.r0; r0 < x.r1 && ok; r0 += ATT_TILE, ++n) {
        // this lane's row: tile row gw*32 + lane
        const int rr = r0 + gw * 32 + lane;
        const uint8_t* src = nullptr;        // bf16 row, or e4m3 nope row
        const __nv_bfloat16* rsrc = nullptr; // mixed: rope row
        float rscale = 0.f;
        long long pos = 0;
        if (rr < x.r1) {
          if (rr < x.nsel) {
            int s = a.idx ? __ldg(a.idx + ((size_t)x.b * a.Tq + x.i) * a.k + rr) : rr;
            if (s >= a.N) { csa_flag_error(ERRBIT_BAD_INDEX); s = -1; }
            const long long prow = s >= 0 ? page_row(a.ent_pg, x.b, s, a.N) : -1;
            if (s >= 0 && prow < 0) csa_flag_error(ERRBIT_BAD_INDEX);   // block outside the pool
            if (prow >= 0) {
              const size_t row = (size_t)prow;
              if (a.kv_mixed) {
                src = reinterpret_cast<const uint8_t*>(a.ent) + row * (ATT_D - ATT_R);
                rsrc = a.ent_rope + row * ATT_R;
                rscale = __ldg(a.ent_scale + row);
              } else {
                src = reinterpret_cast<const uint8_t*>(a.ent) + row * ATT_D * 2;
              }
              pos = a.ent_rotated ? 0 : (long long)a.m * (s + 1) - 1;   // rotated already: turn by -t only
            }
          } else {
            const long long tok = x.w0 + (rr - x.nsel);
            const long long prow =
                (tok >= x.wbase && tok < x.wbase + a.T_win)
                    ? page_row(a.win_pg, x.b, window_row(a.win_pg, tok, x.wbase, a.T_win), a.T_win)
                    : -1;
            if (prow >= 0) {
              const size_t row = (size_t)prow;
              if (a.kv_mixed) {
                src = reinterpret_cast<const uint8_t*>(a.win) + row * (ATT_D - ATT_R);
                rsrc = a.win_rope + row * ATT_R;
                rscale = __ldg(a.win_scale + row);
              } else {
                src = reinterpret_cast<const uint8_t*>(a.win) + row * ATT_D * 2;
              }
              pos = tok;
            } else {
              csa_flag_error(ERRBIT_BAD_INDEX);   // outside this batch row's window buffer or pool
            }
          }
        }
        if (n == (uint32_t)CSA_TRACE_TILE && gw == 0 && lane == 0) CSA_TRACE_MARK(5);
        // rows with no source (past the chunk, index -1) take logit -inf in the softmax
        {
          const uint32_t bits = __ballot_sync(0xffffffffu, src != nullptr);
          if (lane == 0) rmask[(n & 1) * 4 + gw] = bits;
        }
        if (!a.kv_mixed) {
          // bf16 rows by cp.async: lane l copies 16-byte granule (l & 7) of rows
          // (l >> 3) + 4k, k < 8, of this warp's 32, straight into the swizzled tile.
          // Each lane's copies of chunk c arrive on the chunk's barrier when they land
          // (the barrier's pending count rises by one per lane until then); rows
          // without a source are zero-filled and masked above.
          const uint8_t* rsrc8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            rsrc8[k] = reinterpret_cast<const uint8_t*>(
                __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(src), (lane >> 3) + 4 * k));
          auto cp_chunk = [&](int c) {
            const int u = lane & 7;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int tr = gw * 32 + (lane >> 3) + 4 * k;
              const uint8_t* sp = rsrc8[k];
              cp_async16(smem_u32(sE + c * 16384 + tr * 128 + ((u ^ (tr & 7)) << 4)),
                         sp ? sp + c * 128 + u * 16 : reinterpret_cast<const uint8_t*>(a.q), sp != nullptr);
            }
            if (!(c == 7 && a.rotate_rows)) {        // chunk 7 is released after its RoPE below
              cp_async_mbar_arrive(chunk_full + c);
              __syncwarp();
              if (lane == 0) mbar_arrive(chunk_full + c);
            }
          };
          if (r0 == x.r0) {
            // first tile of the item: every chunk pair is free once the last PV of
            // the previous item is done; fetch each row's 1 KB together
            for (int c2 = 0; c2 < 4 && ok; ++c2)
              if (!mbar_wait(chunk_free + c2, (n & 1) ^ 1, abort_flag)) ok = false;
            if (!ok) break;
            for (int c = 0; c < 8; ++c) cp_chunk(c);
            __syncwarp();
            if (n == (uint32_t)CSA_TRACE_TILE && gw == 0 && lane == 0) CSA_TRACE_MARK(6);
            if (!a.rel_rope) {
              // absolute-RoPE mode: rotate this warp's 16 heads of the TMA-loaded
              // queries (chunk 7 = dims 448..511) at t, then release them to the MMA
              if (!mbar_wait(q_full, nitem & 1, abort_flag)) { ok = false; break; }
              ++nitem;
#pragma unroll
              for (int k2 = 0; k2 < 4; ++k2) {
                const int h = gw * 16 + k2 * 4 + (lane >> 3), u = lane & 7;
                uint4* ptr = reinterpret_cast<uint4*>(sQ + 7 * 8192 + h * 128 + ((u ^ (h & 7)) << 4));
                *ptr = rope_unit(*ptr, x.t, ropeF, u * 4);
              }
              fence_proxy_async();
              __syncwarp();
              if (lane == 0) mbar_arrive(q_ready);
            }
          } else {
            // later tiles: each chunk pair as soon as the PV block that read it is done
            for (int c2 = 0; c2 < 4 && ok; ++c2) {
              if (!mbar_wait(chunk_free + c2, (n & 1) ^ 1, abort_flag)) { ok = false; break; }
              cp_chunk(2 * c2);
              cp_chunk(2 * c2 + 1);
            }
            if (!ok) break;
          }
          if (a.rotate_rows) {
            // RoPE of this warp's 32 rows once its chunk 7 (dims 448..511) has landed
            cp_async_commit();                        // wait for every copy this lane issued
            cp_async_wait<0>();
            __syncwarp();
            if (n == (uint32_t)CSA_TRACE_TILE && gw == 0 && lane == 0) CSA_TRACE_MARK(7);
            uint8_t* c7 = sE + 7 * 16384;
#pragma unroll 2
            for (int k2 = 0; k2 < 8; ++k2) {
              const int rl = k2 * 4 + (lane >> 3);
              const int u = lane & 7;
              const long long p = __shfl_sync(0xffffffffu, pos, rl) - (a.rel_rope ? x.t : 0);
              const int tr = gw * 32 + rl;
              uint4* ptr = reinterpret_cast<uint4*>(c7 + tr * 128 + ((u ^ (tr & 7)) << 4));
              *ptr = rope_unit(*ptr, p, ropeF, u * 4);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(chunk_full + 7);
            if (n == (uint32_t)CSA_TRACE_TILE && gw == 0 && lane == 0) CSA_TRACE_MARK(8);
          }
          continue;
        }
        // ---- FP8 / BF16-RoPE rows (kv_mixed) ----
        // Every copy of the tile goes out at once: the 64 e4m3 bytes of each
        // 64-dim chunk (0..6) land in the upper half of the row's 128-byte
        // slot, the RoPE dims (chunk 7) land as bf16 in place.  The e4m3 bytes
        // are then widened to bf16 in place (times the row scale).
        for (int c2 = 0; c2 < 4 && ok; ++c2)
          if (!mbar_wait(chunk_free + c2, (n & 1) ^ 1, abort_flag)) ok = false;
        if (!ok) break;
#pragma unroll 1
        for (int c = 0; c < 7; ++c) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int rl = (k * 32 + lane) >> 2, u4 = lane & 3;
            const uint8_t* s_row = reinterpret_cast<const uint8_t*>(
                __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(src), rl));
            const uint32_t dst = smem_u32(sE + c * 16384 + (gw * 32 + rl) * 128 + 64 + u4 * 16);
            cp_async16(dst, s_row ? s_row + c * 64 + u4 * 16 : reinterpret_cast<const uint8_t*>(a.q),
                       s_row != nullptr);
          }
        }
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) {
          const int rl = k2 * 4 + (lane >> 3), u = lane & 7;
          const uint8_t* r_row = reinterpret_cast<const uint8_t*>(
              __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(rsrc), rl));
          const int tr = gw * 32 + rl;
          const uint32_t dst = smem_u32(sE + 7 * 16384 + tr * 128 + ((u ^ (tr & 7)) << 4));
          cp_async16(dst, r_row ? r_row + u * 16 : reinterpret_cast<const uint8_t*>(a.q), r_row != nullptr);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < 7; ++c) {
          uint2 raw[8];
#pragma unroll
          for (int k2 = 0; k2 < 8; ++k2) {
            const int tr = gw * 32 + k2 * 4 + (lane >> 3);
            raw[k2] = *reinterpret_cast<const uint2*>(sE + c * 16384 + tr * 128 + 64 + (lane & 7) * 8);
          }
          __syncwarp();                                // every row's bytes read before any is overwritten
#pragma unroll
          for (int k2 = 0; k2 < 8; ++k2) {
            const int rl = k2 * 4 + (lane >> 3), u = lane & 7;
            const float sc = __shfl_sync(0xffffffffu, rscale, rl);
            const int tr = gw * 32 + rl;
            *reinterpret_cast<uint4*>(sE + c * 16384 + tr * 128 + ((u ^ (tr & 7)) << 4)) =
                e4m3x8_to_bf16(raw[k2], sc);
          }
          __syncwarp();
        }
        {
          // RoPE of this warp's 32 rows: chunk 7 holds dims 448..511
          uint8_t* c7 = sE + 7 * 16384;
#pragma unroll 2
          for (int k2 = 0; k2 < 8; ++k2) {
            const int rl = k2 * 4 + (lane >> 3);
            const int u = lane & 7;
            const long long p = __shfl_sync(0xffffffffu, pos, rl) - (a.rel_rope ? x.t : 0);
            const int tr = gw * 32 + rl;
            uint4* ptr = reinterpret_cast<uint4*>(c7 + tr * 128 + ((u ^ (tr & 7)) << 4));
            *ptr = rope_unit(*ptr, p, ropeF, u * 4);
          }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0)
          for (int c = 0; c < 8; ++c) mbar_arrive(chunk_full + c);
      }
    }
  } else if (warp == 8) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16(ATT_TILE, ATT_HG);
      const uint32_t id_pv = idesc_bf16(ATT_TILE, ATT_HG) | (1u << 15) | (1u << 16);
      uint32_t n = 0, nitem = 0;
      bool ok = true;
      const uint32_t e_base = smem_u32(sE), q_base = smem_u32(sQ), p_base = smem_u32(sP);
      for (int it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
        const AttRow x = att_item(a, it);
        if (nitem == 0) CSA_TRACE_MARK(29);
        if (x.r1 <= x.r0) continue;
        {
          // queries of this head group: 8 boxes of [64 heads x 64 dims], 128-byte swizzled
          if (!mbar_wait(q_free, (nitem & 1) ^ 1, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(q_full, ATT_HG * ATT_D * 2);
          const int qrow = (x.b * a.Tq + x.i) * a.n_h + x.hg * ATT_HG;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            tma_load_3d(sQ + c * 8192, &tm_q, q_full, c * 64, qrow, 0);
            if (nitem == 0 && c == 0) CSA_TRACE_MARK(30);
          }
          if (nitem == 0) CSA_TRACE_MARK(3);
        }
        if (!mbar_wait(a.rel_rope ? q_full : q_ready, nitem & 1, abort_flag)) { ok = false; break; }
        if (nitem == 0) CSA_TRACE_MARK(4);
        const uint32_t item = nitem++;
        int j = 0;
        for (int r0 = x.r0; r0 < x.r1; r0 += ATT_TILE, ++n, ++j) {
          const uint32_t sb = n & 1;
          if (!mbar_wait(s_free + sb, ((n >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
          // S^T = E * Q^T over the 8 dim chunks as they land
          for (int c = 0; c < 8; ++c) {
            if (!mbar_wait(chunk_full + c, n & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = sdesc_sw128(e_base + c * 16384 + kk * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(q_base + c * 8192 + kk * 32, 16, 1024);
              umma_f16(tmem + TM_S + sb * ATT_HG, ad, bd, id_qk, (c | kk) ? 1u : 0u);
            }
          }
          if (!ok) break;
          if (n == (uint32_t)CSA_TRACE_TILE) CSA_TRACE_MARK(9);
          umma_commit(s_full + sb);
          if (r0 + ATT_TILE >= x.r1) umma_commit(q_free);
          if (j == 0 && !mbar_wait(o_free, (item & 1) ^ 1, abort_flag)) { ok = false; break; }
          if (!mbar_wait(p_full, n & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          // O^T[dims block bk] += E^T * P^T
          for (int bk = 0; bk < 4; ++bk) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t ad = sdesc_sw128(e_base + bk * 32768 + kk * 2048, 16384, 1024);
              const uint64_t bd = sdesc_sw128(p_base + kk * 2048, 8192, 1024);
              umma_f16(tmem + TM_O + bk * ATT_HG, ad, bd, id_pv, (j > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(chunk_free + bk);
          }
          umma_commit(p_free);
          if (n == (uint32_t)CSA_TRACE_TILE) CSA_TRACE_MARK(12);
        }
      }
      umma_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else {
    // ======================= softmax / epilogue (warps 0-3) =======================
    const int q4 = warp;                              // TMEM lane quarter
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    float* my_m = mrow + q4 * 64;
    float* my_f = facs + q4 * 64;
    uint32_t n = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
      const AttRow x = att_item(a, it);
      float m_run[2] = {-INFINITY, -INFINITY};        // heads 2*lane, 2*lane+1
      float l_run[2] = {0.f, 0.f};
      int j = 0;
      for (int r0 = x.r0; r0 < x.r1; r0 += ATT_TILE, ++n, ++j) {
        const uint32_t sb = n & 1, par = n & 1;
        if (!mbar_wait(s_full + sb, (n >> 1) & 1, abort_flag)) { ok = false; break; }
        if (n == (uint32_t)CSA_TRACE_TILE && q4 == 0 && lane == 0) CSA_TRACE_MARK(10);
        tc_fence_after();
        float xs[64];
        {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + TM_S + sb * ATT_HG, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) xs[e] = __uint_as_float(r[e]);
          tmem_ld32(tmem + lane_base + TM_S + sb * ATT_HG + 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) xs[32 + e] = __uint_as_float(r[e]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free + sb);
        if (n == (uint32_t)CSA_TRACE_TILE && q4 == 0 && lane == 0) CSA_TRACE_MARK(23);
        const bool valid = (rmask[(n & 1) * 4 + q4] >> lane) & 1u;
#pragma unroll
        for (int e = 0; e < 64; ++e) xs[e] = valid ? xs[e] * a.scale_log2 : -INFINITY;
        // ---- per-head tile max over the 128 rows ----
        float red[32];
        warp_reduce_scatter64_from<true>([&](int e) { return xs[e]; }, red, lane);
        maxp[(par * 4 + q4) * 64 + 2 * lane] = red[0];
        maxp[(par * 4 + q4) * 64 + 2 * lane + 1] = red[1];
        __syncwarp();
        if (lane == 0) mbar_arrive(grp_a);
        if (!mbar_wait(grp_a, par, abort_flag)) { ok = false; break; }
        if (n == (uint32_t)CSA_TRACE_TILE && q4 == 0 && lane == 0) CSA_TRACE_MARK(24);
        bool resc = false;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * lane + e;
          float tm = maxp[(par * 4 + 0) * 64 + h];
          tm = fmaxf(tm, maxp[(par * 4 + 1) * 64 + h]);
          tm = fmaxf(tm, maxp[(par * 4 + 2) * 64 + h]);
          tm = fmaxf(tm, maxp[(par * 4 + 3) * 64 + h]);
          float f = 1.f;
          if (j == 0) {
            m_run[e] = tm;
          } else if (tm > m_run[e] + ATT_TAU) {
            f = exp2f(m_run[e] - tm);
            m_run[e] = tm;
            resc = true;
          }
          my_m[h] = m_run[e];
          my_f[h] = f;
          l_run[e] *= f;
        }
        resc = __any_sync(0xffffffffu, resc);
        __syncwarp();
        // ---- P = exp2(x - m), bf16; row pieces of P^T ----
        // (a head whose rows so far are all masked has m = -inf: its P is 0, not NaN)
        // (the row sums are taken later from the same bf16-rounded P, unpacked)
        uint32_t pk[32];
        const float2* mm = reinterpret_cast<const float2*>(my_m);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float2 m2 = mm[e];
          const float p0 = ex2_approx(xs[2 * e] - (m2.x == -INFINITY ? 0.f : m2.x));
          const float p1 = ex2_approx(xs[2 * e + 1] - (m2.y == -INFINITY ? 0.f : m2.y));
          pk[e] = pack_bf16x2(p0, p1);
        }
        if (n == (uint32_t)CSA_TRACE_TILE && q4 == 0 && lane == 0) CSA_TRACE_MARK(25);
        // PV of the previous tile must be done before P^T and O^T are touched
        if (!mbar_wait(p_free, (n & 1) ^ 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        {
          const int tr = q4 * 32 + lane;
          uint8_t* prow = sP + tr * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(prow + ((u ^ (tr & 7)) << 4)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
        if (resc && j > 0) {
          // O^T columns (heads) times their factors; this warp owns dims rows
          // q4*32 + lane of each 128-dim block.  Eight columns at a time: the
          // packed P words stay live across this rare path.
#pragma unroll 1
          for (int cc = 0; cc < 4 * ATT_HG; cc += 8) {
            uint32_t r[8];
            const uint32_t ta = tmem + lane_base + TM_O + cc;
            tmem_ld8(ta, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 8; ++e)
              r[e] = __float_as_uint(__uint_as_float(r[e]) * my_f[(cc & (ATT_HG - 1)) + e]);
            tmem_st8(ta, r);
          }
          tmem_st_wait();
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        if (n == (uint32_t)CSA_TRACE_TILE && q4 == 0 && lane == 0) CSA_TRACE_MARK(11);
        // ---- per-head row sums (of the bf16-rounded P the MMA used) ----
        float sr[32];
        warp_reduce_scatter64_from<false>([&](int e) {
          const uint32_t w = pk[e >> 1];
          return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
        }, sr, lane);
        sump[(par * 4 + q4) * 64 + 2 * lane] = sr[0];
        sump[(par * 4 + q4) * 64 + 2 * lane + 1] = sr[1];
        __syncwarp();
        if (lane == 0) mbar_arrive(grp_b);
        if (!mbar_wait(grp_b, par, abort_flag)) { ok = false; break; }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * lane + e;
          l_run[e] += sump[(par * 4 + 0) * 64 + h] + sump[(par * 4 + 1) * 64 + h] +
                      sump[(par * 4 + 2) * 64 + h] + sump[(par * 4 + 3) * 64 + h];
        }
        if (n == (uint32_t)CSA_TRACE_TILE && q4 == 0 && lane == 0) CSA_TRACE_MARK(13);
      }
      if (!ok) break;
      // ======================= item epilogue =======================
      const bool single = (a.nch == 1);
      // split item and one item per CTA: the entry tile is free for staging
      const bool stage_out = !single && (int)gridDim.x >= a.items;
      if (j > 0) {
        if (!mbar_wait(p_free, (n - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
      }
      if (it == (int)blockIdx.x && q4 == 0 && lane == 0) CSA_TRACE_MARK(14);
      if (a.cl_reduce) {
        // cluster merge (one item per CTA): only this chunk's (max, sum) is
        // recorded here; the merge after the role loops moves O out of TMEM
        float* ml = reinterpret_cast<float*>(smem + AttSmem::ML);
        if (q4 == 0) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            ml[(2 * lane + e) * 2] = m_run[e];
            ml[(2 * lane + e) * 2 + 1] = j > 0 ? l_run[e] : 0.f;
          }
          if (lane == 0) reinterpret_cast<int*>(smem + AttSmem::MISC)[2] = j > 0 ? 1 : 0;
        }
        continue;
      }
      // per-head output scale into this warp's table
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * lane + e;
        if (single) {
          const float zs = __ldg(a.sink + x.hg * ATT_HG + h) * 1.4426950408889634f;
          const float M = fmaxf(m_run[e], zs);
          const float den = l_run[e] * exp2f(m_run[e] - M) + exp2f(zs - M);
          my_f[h] = exp2f(m_run[e] - M) / den;
        } else {
          my_f[h] = 1.f;
          float* ml = a.cl_reduce ? reinterpret_cast<float*>(smem + AttSmem::ML) + h * 2
                                  : a.part_ml + ((size_t)it * ATT_HG + h) * 2;
          if (q4 == 0) { ml[0] = m_run[e]; ml[1] = l_run[e]; }
        }
      }
      __syncwarp();
      const size_t orow = ((size_t)x.b * a.Tq + x.i) * a.n_h + (size_t)x.hg * ATT_HG;
#pragma unroll 1
      for (int bk = 0; bk < 4; ++bk) {
        const int dim = bk * 128 + q4 * 32 + lane;
        float c = 1.f, s = 0.f;
        const bool rope_dim = dim >= ATT_D - ATT_R;
        const bool rot_out = single && rope_dim && !a.rel_rope;
        if (rot_out) rope_cos_sin(-x.t, ropeF[(dim - (ATT_D - ATT_R)) >> 1], c, s);
        uint32_t r2[64];
        if (j > 0) {
          tmem_ld32(tmem + lane_base + TM_O + bk * ATT_HG, r2);
          tmem_ld32(tmem + lane_base + TM_O + bk * ATT_HG + 32, r2 + 32);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) r2[e] = 0u;
        }
#pragma unroll
        for (int hh = 0; hh < 64; hh += 32) {
          const uint32_t* r = r2 + hh;
          if (single) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              float v = __uint_as_float(r[e]) * my_f[hh + e];
              const float pv = __shfl_xor_sync(0xffffffffu, v, 1);
              if (rot_out) v = (lane & 1) ? (pv * s + v * c) : (v * c - pv * s);
              a.out[(orow + hh + e) * ATT_D + dim] = __float2bfloat16_rn(v);
            }
          } else if (stage_out) {
            // unnormalised partial into the staging copy of its global layout
            // [64 heads][512 dims]: consecutive lanes write consecutive dims
            float* st = reinterpret_cast<float*>(sE) + dim;
#pragma unroll
            for (int e = 0; e < 32; ++e) st[(size_t)(hh + e) * ATT_D] = __uint_as_float(r[e]);
          } else {
            // unnormalised partial, layout [item][64 heads][512 dims]
            float* dst = a.part_o + (size_t)it * ATT_HG * ATT_D + dim;
#pragma unroll
            for (int e = 0; e < 32; ++e) dst[(size_t)(hh + e) * ATT_D] = __uint_as_float(r[e]);
          }
        }
      }
      if (stage_out && !a.cl_reduce) {
        // one bulk copy of the staged 128 KB partial to global memory
        fence_proxy_async();
        named_bar_sync(2, 128);
        if (threadIdx.x == 0) {
          asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                           a.part_o + (size_t)it * ATT_D * ATT_HG),
                       "r"(smem_u32(sE)), "r"(ATT_D * ATT_HG * 4)
                       : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && j > 0) mbar_arrive(o_free);
      if (it == (int)blockIdx.x && q4 == 0 && lane == 0) CSA_TRACE_MARK(15);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) CSA_TRACE_MARK(16);
  if (a.cl_reduce) attend_cluster_merge(a, smem, tmem, merge_bar, ml_bar);
  if (warp == 8) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0) { CSA_TRACE_MARK(22); CSA_TRACE_WALL(21); }
}

// ----------------------------------------------------------------------------
// split-chunk combine: out[b,i,h,:] = sum_c 2^(m_c - M) O_c / (sum_c 2^(m_c - M) l_c
// + 2^(z'_h log2 e - M)), then (absolute-RoPE mode) the RoPE dims rotated back by -t.
// Partials are [chunk][64 heads][512 dims] f32.  One CTA per (query row, head
// group, 8 output dims): thread pairs read a head's 32-byte slice of every
// chunk and write one 16-byte bf16 run.
// ----------------------------------------------------------------------------
struct CombineArgs {
  const float* part_o; const float* part_ml; const float* sink;
  __nv_bfloat16* out;
  const int32_t* q_pos;           // [B, Tq] (null: t = i)
  int Tq, n_h, HG, nch;
  int rel_rope;       // 1 = output already relative to t (no rotation)
  RopeFreqs rf;
};

constexpr int CMB_THREADS = 128;
constexpr int CMB_DIMS = 8;                        // output dims per CTA

__global__ void __launch_bounds__(CMB_THREADS) attend_combine_kernel(const CombineArgs a) {
  pdl_enter();
  extern __shared__ float cmb_w[];                 // [nch][64][2]: (m, l), then weights
  const int db = (blockIdx.x % (ATT_D / CMB_DIMS)) * CMB_DIMS;
  const int unit = blockIdx.x / (ATT_D / CMB_DIMS);   // (b * Tq + i) * HG + hg
  const int hg = unit % a.HG;
  const int bi = unit / a.HG;
  const int i = bi % a.Tq;
  const size_t it0 = (size_t)unit * a.nch;
  const int tid = threadIdx.x;
  // every chunk's (m, l) of this unit: one contiguous run, all loads in flight
  {
    const float4* src = reinterpret_cast<const float4*>(a.part_ml + it0 * ATT_HG * 2);
    float4* dst = reinterpret_cast<float4*>(cmb_w);
    for (int e = tid; e < a.nch * ATT_HG / 2; e += CMB_THREADS) dst[e] = __ldg(src + e);
  }
  __syncthreads();
  if (tid < ATT_HG) {
    const int h = tid;
    const float zs = __ldg(a.sink + hg * ATT_HG + h) * 1.4426950408889634f;
    float M = zs;
    for (int c = 0; c < a.nch; ++c) M = fmaxf(M, cmb_w[(c * ATT_HG + h) * 2]);
    float den = exp2f(zs - M);
    for (int c = 0; c < a.nch; ++c) {
      const float mc = cmb_w[(c * ATT_HG + h) * 2];
      if (mc != -INFINITY) den += cmb_w[(c * ATT_HG + h) * 2 + 1] * exp2f(mc - M);
    }
    const float inv = 1.f / den;
    for (int c = 0; c < a.nch; ++c) {
      const float mc = cmb_w[(c * ATT_HG + h) * 2];
      cmb_w[(c * ATT_HG + h) * 2] = mc == -INFINITY ? 0.f : exp2f(mc - M) * inv;   // weight
    }
  }
  __syncthreads();
  // thread: head tid / 2, dims db + 4 (tid & 1) .. + 3
  const int h = tid >> 1, half = tid & 1;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* src = a.part_o + (it0 * ATT_HG + h) * ATT_D + db + 4 * half;
  for (int c = 0; c < a.nch; ++c) {
    const float w = cmb_w[(c * ATT_HG + h) * 2];
    const float4 v = __ldg(reinterpret_cast<const float4*>(src + (size_t)c * ATT_HG * ATT_D));
    acc.x += v.x * w; acc.y += v.y * w; acc.z += v.z * w; acc.w += v.w * w;
  }
  float v8[CMB_DIMS];
  v8[0] = acc.x; v8[1] = acc.y; v8[2] = acc.z; v8[3] = acc.w;
  v8[4] = __shfl_down_sync(0xffffffffu, acc.x, 1);
  v8[5] = __shfl_down_sync(0xffffffffu, acc.y, 1);
  v8[6] = __shfl_down_sync(0xffffffffu, acc.z, 1);
  v8[7] = __shfl_down_sync(0xffffffffu, acc.w, 1);
  if (half == 0) {
    if (!a.rel_rope && db >= ATT_D - ATT_R) {
      const long long t = query_pos(a.q_pos, bi, i);
#pragma unroll
      for (int p = 0; p < CMB_DIMS / 2; ++p) {
        float cs, sn;
        rope_cos_sin(-t, a.rf.F[((db - (ATT_D - ATT_R)) >> 1) + p], cs, sn);
        const float x0 = v8[2 * p], x1 = v8[2 * p + 1];
        v8[2 * p] = x0 * cs - x1 * sn;
        v8[2 * p + 1] = x0 * sn + x1 * cs;
      }
    }
    __nv_bfloat16* o = a.out + ((size_t)bi * a.n_h + (size_t)hg * ATT_HG + h) * ATT_D + db;
    *reinterpret_cast<uint4*>(o) = f_to_bf16x8(v8);
  }
}

// ----------------------------------------------------------------------------
// RoPE pre-rotation of a row set (bf16 rows, rotated copy of the last 64 dims
// at each row's position): used when many query rows gather the same rows.
// ----------------------------------------------------------------------------
struct RotateArgs {
  const __nv_bfloat16* src; __nv_bfloat16* dst;
  long long rows;                 // B * rows per batch row
  int rows_per_b;
  int m;                          // >0: compressed entries (pos = m(s+1)-1); 0: tokens
  const int32_t* base;            // tokens: [B] token position of each batch row's row 0 (null: 0)
  RowPages pg;                    // row map of src; dst is always flat (logical order)
  RopeFreqs rf;
};

__global__ void __launch_bounds__(256) rope_rotate_rows_kernel(const RotateArgs a) {
  __shared__ unsigned long long F[64];          // lanes read different frequencies
  if (threadIdx.x < 64) F[threadIdx.x] = a.rf.F[threadIdx.x];
  __syncthreads();
  pdl_enter();
  // one thread per 16-byte unit; 64 units per 512-dim row
  const long long u_all = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u_all >= a.rows * 64) return;
  const long long row = u_all >> 6;               // logical: b * rows_per_b + s
  const int u = (int)(u_all & 63);
  const int b = (int)(row / a.rows_per_b);
  const long long s = row - (long long)b * a.rows_per_b;
  const long long pos = a.m > 0 ? (long long)a.m * (s + 1) - 1 : window_base(a.base, b) + s;
  // source row: entry s, or the window row that holds token pos
  const long long j = (a.m == 0 && a.pg.ring) ? (pos >= 0 ? pos % a.rows_per_b : -1) : s;
  const long long src = j >= 0 ? page_row(a.pg, b, j, a.rows_per_b) : -1;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (src >= 0) {
    v = __ldg(reinterpret_cast<const uint4*>(a.src + src * ATT_D + u * 8));
    if (u >= (ATT_D - ATT_R) / 8) v = rope_unit(v, pos, F, (u - (ATT_D - ATT_R) / 8) * 4);
  } else if (j >= 0 && u == 0) {
    csa_flag_error(ERRBIT_BAD_INDEX);             // block outside the pool
  }
  *reinterpret_cast<uint4*>(a.dst + row * ATT_D + u * 8) = v;
}

}  // namespace csa
