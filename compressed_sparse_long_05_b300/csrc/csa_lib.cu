// C ABI of the CSA / HCA forward kernels (declared in include/csa.h).
//
// One translation unit: the kernels live in the included .cuh files so that
// they share the device error word without relocatable device code.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/csa.h"
#include "common.cuh"
#include "compress.cuh"
#include "topk.cuh"
#include "topk2.cuh"
#include "simt_f32.cuh"
#include "index_tc.cuh"
#include "index_fp4.cuh"
#include "attend_tc.cuh"
#include "gemm_tc.cuh"

#include <cudaTypedefs.h>

namespace {

thread_local char g_cuda_msg[256] = "";

csa_status_t cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_cuda_msg, sizeof(g_cuda_msg), "%s: %s", where, cudaGetErrorString(e));
  return CSA_ERR_CUDA;
}

#define CSA_CHECK_LAUNCH(where)                          \
  do {                                                   \
    cudaError_t e_ = cudaGetLastError();                 \
    if (e_ != cudaSuccess) return cuda_fail(e_, where);  \
  } while (0)

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }

RopeFreqs make_rope(int r, float base) {
  RopeFreqs rf;
  memset(&rf, 0, sizeof(rf));
  rf.half = r / 2;
  const double two_pi = 6.283185307179586476925286766559;
  for (int j = 0; j < r / 2; ++j) {
    const double theta = std::pow((double)base, -2.0 * j / (double)r);
    const double frac = theta / two_pi;                 // revolutions per position, < 1
    rf.F[j] = (unsigned long long)std::ldexp(frac, 64);
  }
  return rf;
}

int sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}


// Programmatic stream serialisation lets a kernel's CTAs launch while the
// previous kernel in the stream still runs: every kernel here sets up its
// barriers and tensor memory, then waits on the grid dependency before its
// first global memory access, so the setting never changes results.  Off:
// applied to every launch it made the decode step slower (128K: 69 vs 59 us,
// early grids took the SMs the running one's clusters needed), and applied
// only inside one layer forward (index -> top-k -> attention) the launch gaps
// vanished but the early grids waited as long (63.4 vs 67.0 us per step).
// Measured again on the current kernels: for the selector after the index
// kernel still slower (decode 128K 46.9 -> 53.5 us); for the attention kernel
// faster on short launches (HCA decode at 1M 30.15 -> 28.6 us, CSA decode at
// 128K 46.69 -> 46.55 us) but slower on the persistent prefill launches
// (CSA prefill 32K attention 22.25 -> 23.3 ms, HCA prefill 64K 21.9 -> 23.2
// ms), so attention launches of at most kProgrammaticAttendItems work items
// per CTA take it.
constexpr bool kProgrammaticLaunch = false;
constexpr int kProgrammaticAttendItems = 4;

// As launch_ex, with programmatic serialisation against the previous kernel when `pdl`.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          int cluster, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Launch with an optional cluster size (and programmatic serialisation when on).
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      int cluster, Args... args) {
  return launch_ex_pdl(kern, grid, block, smem, st, cluster, kProgrammaticLaunch, args...);
}


// 3-D bf16 tensor map (x fastest), 128-byte swizzle, zero fill out of bounds.
bool tmap_bf16_3d(CUtensorMap* m, const void* base, uint64_t x, uint64_t y, uint64_t z,
                  uint64_t y_stride_bytes, uint64_t z_stride_bytes, uint32_t box_x, uint32_t box_y) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {x, y, z};
  cuuint64_t strides[2] = {y_stride_bytes, z_stride_bytes};
  cuuint32_t box[3] = {box_x, box_y, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 tensor map with a full 3-D box, 128-byte swizzle, zero fill.
bool tmap_bf16_3d_box(CUtensorMap* m, const void* base, const uint64_t dims_[3],
                      const uint64_t strides_[2], const uint32_t box_[3]) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {dims_[0], dims_[1], dims_[2]};
  cuuint64_t strides[2] = {strides_[0], strides_[1]};
  cuuint32_t box[3] = {box_[0], box_[1], box_[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D byte tensor map (x fastest, 64-byte rows), 64-byte swizzle, zero fill.
bool tmap_u8_3d_sw64(CUtensorMap* m, const void* base, uint64_t x, uint64_t y, uint64_t z,
                     uint64_t y_stride, uint64_t z_stride, uint32_t box_y) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {x, y, z};
  cuuint64_t strides[2] = {y_stride, z_stride};
  cuuint32_t box[3] = {(cuuint32_t)x, box_y, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 1-D map over `n` 8-byte elements (one element = the 8 scale bytes of a row).
bool tmap_u64_1d(CUtensorMap* m, const void* base, uint64_t n, uint32_t box) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[1] = {n};
  cuuint64_t strides[1] = {8};
  cuuint32_t boxd[1] = {box};
  cuuint32_t estr[1] = {1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 1, const_cast<void*>(base), dims, strides,
                   boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Work split of the persistent index kernels: query groups of QT rows; when
// there are fewer (batch row, group) pairs than SMs, the entry tiles of a
// group are cut into chunks so that every SM streams part of K.
csa_status_t plan_index(csa::IndexTcArgs& a, int QT, int B, int Tq, int N) {
  a.QT = QT > Tq ? Tq : QT;
  a.G = (Tq + a.QT - 1) / a.QT;
  a.tiles_max = (N + csa::IDX_TILE - 1) / csa::IDX_TILE;
  const int sms = sm_count();
  const long long units = (long long)B * a.G;
  if (units >= sms) {
    a.chunk_tiles = a.tiles_max;
  } else {
    // at most `sms` items: floor(sms / units) chunks per unit, so no SM takes two
    const long long per_unit = sms / units;
    a.chunk_tiles = (int)((a.tiles_max + per_unit - 1) / per_unit);
    if (a.chunk_tiles < 1) a.chunk_tiles = 1;
  }
  a.chunks = (a.tiles_max + a.chunk_tiles - 1) / a.chunk_tiles;
  long long items = units * a.chunks;
  if (items > 0x7fffffff) return CSA_ERR_UNSUPPORTED;
  a.items = (int)items;
  return CSA_OK;
}

// Host checks of a row map (csa_pages_t) into its device form.  rows: logical
// rows per sequence the call may read; ring_ok: window rows; pow2: tiled key
// loads need block_rows a power of two >= 8.
csa_status_t check_pages(const csa_pages_t* p, long long rows, bool ring_ok, bool pow2,
                         RowPages* out) {
  memset(out, 0, sizeof(*out));
  out->shift = -1;
  if (!p) return CSA_OK;
  if (p->ring && !ring_ok) return CSA_ERR_INVALID_ARG;
  out->ring = p->ring ? 1 : 0;
  if (!p->block_table) return CSA_OK;
  if (!aligned(p->block_table, 4) || p->block_rows < 1 || p->num_blocks < 1 || p->max_blocks < 1)
    return CSA_ERR_INVALID_ARG;
  if ((rows + p->block_rows - 1) / p->block_rows > p->max_blocks) return CSA_ERR_INVALID_ARG;
  if ((long long)p->num_blocks * p->block_rows >= 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
  if (pow2 && (p->block_rows < 8 || (p->block_rows & (p->block_rows - 1)))) return CSA_ERR_UNSUPPORTED;
  out->table = p->block_table;
  out->max_blocks = p->max_blocks;
  out->block_rows = p->block_rows;
  out->num_blocks = p->num_blocks;
  out->shift = -1;
  if ((p->block_rows & (p->block_rows - 1)) == 0) {
    out->shift = 0;
    while ((1 << out->shift) < p->block_rows) ++out->shift;
  }
  return CSA_OK;
}

template <int H>
csa_status_t launch_index_fp4(const void* qI, const void* qI_sf, const float* w, const void* K,
                              const void* K_sf, const RowPages& kpg, const int32_t* q_pos,
                              void* scores, int scores_bf16, int B, int Tq, int N, int m,
                              uint32_t* hist, cudaStream_t stream) {
  csa::IndexFp4Args fa;
  memset(&fa, 0, sizeof(fa));
  csa::IndexTcArgs& a = fa.t;
  a.w = w; a.scores = scores; a.scores_bf16 = scores_bf16; a.q_pos = q_pos;
  a.B = B; a.Tq = Tq; a.N = N; a.m = m;
  csa_status_t st = plan_index(a, 128 / H, B, Tq, N);
  if (st != CSA_OK) return st;
  if ((long long)B * N >= 0x7fffffffLL || (long long)B * Tq * H >= 0x7fffffffLL)
    return CSA_ERR_UNSUPPORTED;
  a.hist = a.QT == 1 ? hist : nullptr;
  const int nqh = a.QT * H;
  a.tmem_cols = 512;
  // accumulator buffers in columns [0, 256), scale factors above; the two
  // epilogue groups take alternate buffers
  a.nbuf = 4 * nqh <= 256 ? 4 : 2;
  CUtensorMap tmK, tmq, tmKs, tmqs;
  bool ok;
  if (kpg.table) {
    // paged keys: maps over the pool, one copy per min(block_rows, 128) rows
    a.k_pg = kpg;
    a.k_piece = kpg.block_rows < csa::IDX_TILE ? kpg.block_rows : csa::IDX_TILE;
    const uint64_t P = (uint64_t)kpg.block_rows, nb = (uint64_t)kpg.num_blocks;
    fa.k_sf = reinterpret_cast<const uint8_t*>(K_sf);   // scale rows by untiled bulk copies
    ok = tmap_u8_3d_sw64(&tmK, K, csa::FP4_ROWB, P, nb, csa::FP4_ROWB, P * csa::FP4_ROWB,
                         (uint32_t)a.k_piece) &&
         tmap_u64_1d(&tmKs, K_sf, P * nb, (uint32_t)a.k_piece);   // prefetched, not copied from
  } else {
    ok = tmap_u8_3d_sw64(&tmK, K, csa::FP4_ROWB, N, B, csa::FP4_ROWB, (uint64_t)N * csa::FP4_ROWB,
                         csa::IDX_TILE) &&
         tmap_u64_1d(&tmKs, K_sf, (uint64_t)B * N, csa::FP4_SF_BOX);
  }
  if (!ok ||
      !tmap_u8_3d_sw64(&tmq, qI, csa::FP4_ROWB, (uint64_t)Tq * H, B, csa::FP4_ROWB,
                       (uint64_t)Tq * H * csa::FP4_ROWB, nqh) ||
      !tmap_u64_1d(&tmqs, qI_sf, (uint64_t)B * Tq * H, nqh))
    return CSA_ERR_UNSUPPORTED;
  const int smem = csa::IndexFp4Smem::BYTES;
  auto kern = csa::index_fp4_kernel<H>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "csa_index fp4 attr");
  const int sms = sm_count();
  const int grid = a.items < sms ? a.items : sms;
  e = launch_ex(kern, dim3(grid), dim3(csa::FP4_THREADS), smem, stream, 1, tmK, tmq, tmKs, tmqs, fa);
  if (e != cudaSuccess) return cuda_fail(e, "csa_index fp4 launch");
  return CSA_OK;
}

template <int H, int C>
csa_status_t launch_index_tc(const void* qI, const float* w, const void* K, const RowPages& kpg,
                             const int32_t* q_pos, void* scores, int scores_bf16, int B, int Tq,
                             int N, int m, uint32_t* hist, cudaStream_t stream,
                             unsigned long long wait_ns = 0, int skip_load_plus1 = 0) {
  csa::IndexTcArgs a;
  memset(&a, 0, sizeof(a));
  a.w = w; a.scores = scores; a.scores_bf16 = scores_bf16; a.q_pos = q_pos;
  a.B = B; a.Tq = Tq; a.N = N; a.m = m;
  a.wait_ns = wait_ns;
  a.skip_load_plus1 = skip_load_plus1;
  csa_status_t st = plan_index(a, 256 / H, B, Tq, N);
  if (st != CSA_OK) return st;
  const int sms = sm_count();
  const int nqh = a.QT * H;
  // four accumulator buffers when they fit: the epilogue of one tile overlaps
  // the MMAs of the next three
  a.nbuf = 4 * nqh <= 512 ? 4 : 2;
  uint32_t cols = 32;
  while (cols < (uint32_t)(a.nbuf * nqh)) cols <<= 1;
  a.tmem_cols = cols;
  CUtensorMap tmK, tmq;
  bool ok;
  if (kpg.table) {
    // paged keys: a map over the pool, one copy per min(block_rows, 128) rows
    a.k_pg = kpg;
    a.k_piece = kpg.block_rows < csa::IDX_TILE ? kpg.block_rows : csa::IDX_TILE;
    ok = tmap_bf16_3d(&tmK, K, C, (uint64_t)kpg.block_rows, (uint64_t)kpg.num_blocks, (uint64_t)C * 2,
                      (uint64_t)kpg.block_rows * C * 2, 64, (uint32_t)a.k_piece);
  } else {
    ok = tmap_bf16_3d(&tmK, K, C, N, B, (uint64_t)C * 2, (uint64_t)N * C * 2, 64, csa::IDX_TILE);
  }
  if (!ok ||
      !tmap_bf16_3d(&tmq, qI, C, (uint64_t)Tq * H, B, (uint64_t)C * 2, (uint64_t)Tq * H * C * 2,
                    64, nqh))
    return CSA_ERR_UNSUPPORTED;
  a.hist = a.QT == 1 ? hist : nullptr;
  a.stages = csa::IndexSmem<H, C>::stages_for(nqh, a.hist != nullptr);
  const int smem = csa::IndexSmem<H, C>(a.stages, nqh, a.hist != nullptr).BYTES;
  auto kern = csa::index_tc_kernel<H, C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "csa_index tc attr");
  const int grid = a.items < sms ? a.items : sms;
  e = launch_ex(kern, dim3(grid), dim3(csa::IDX_THREADS), smem, stream, 1, tmK, tmq, a);
  if (e != cudaSuccess) return cuda_fail(e, "csa_index tc launch");
  return CSA_OK;
}

// Work split and scratch layout of the tensor-core attention path.
struct AttPlan {
  int HG, nch, chunk_rows, items, rotate_rows, rel_rope, cl_reduce;
  int ncs;          // chunks per merging cluster (cl_reduce)
  int cl_partial;   // clusters merge into partials that the combine kernel finishes
  size_t off_part_o, off_part_ml, off_rot_ent, off_rot_win, bytes;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Co-resident clusters of `cl` attention CTAs on the current device (0 when the
// query fails), cached per device and size.
int attend_max_clusters(int cl) {
  static std::mutex mu;
  static int cache_dev = -1;
  static int cache[17];
  int dev = 0;
  if (cl < 2 || cl > 16 || cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache_dev != dev) {
    for (int i = 0; i <= 16; ++i) cache[i] = -1;
    cache_dev = dev;
  }
  if (cache[cl] < 0) {
    int n = 0;
    bool ok = cudaFuncSetAttribute(csa::attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   csa::AttSmem::BYTES) == cudaSuccess;
    if (ok && cl > 8)
      ok = cudaFuncSetAttribute(csa::attend_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
           cudaSuccess;
    if (ok) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)cl);
      cfg.blockDim = dim3(csa::ATT_THREADS);
      cfg.dynamicSmemBytes = csa::AttSmem::BYTES;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = cl;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      ok = cudaOccupancyMaxActiveClusters(&n, csa::attend_tc_kernel, &cfg) == cudaSuccess;
    }
    if (!ok) {
      cudaGetLastError();   // clear the sticky-free error of a failed query
      n = 0;
    }
    cache[cl] = n;
  }
  return cache[cl];
}

// The split is sized for the widest row set any query can have: min(k, N)
// (CSA) or N (HCA) entries plus n_win window tokens.  Queries with fewer rows
// leave their last chunks short or empty.
AttPlan plan_attend(int B, int Tq, int N, int k, int T_win, int n_h, int n_win, int dense,
                    int kv_mixed) {
  AttPlan p;
  memset(&p, 0, sizeof(p));
  p.HG = n_h / csa::ATT_HG;
  const long long nsel = dense ? N : (N < k ? N : k);
  const long long rows_max = nsel + n_win;
  const int tiles = (int)((rows_max + csa::ATT_TILE - 1) / csa::ATT_TILE);
  const long long units = (long long)B * Tq * p.HG;
  const int sms = sm_count();
  int chunk_tiles = tiles;
  if (units < sms && tiles > 1) {
    chunk_tiles = (int)((units * tiles + sms - 1) / sms);
    if (chunk_tiles < 1) chunk_tiles = 1;
  }
  p.nch = (tiles + chunk_tiles - 1) / chunk_tiles;
  if (p.nch < 1) p.nch = 1;
  p.chunk_rows = chunk_tiles * csa::ATT_TILE;
  p.items = (int)(units * p.nch);
  // rotate every stored row once when the queries gather far more rows than exist
  const long long gathered = (long long)B * Tq * rows_max;
  p.rotate_rows = (kv_mixed || gathered <= 2LL * B * ((long long)N + T_win)) ? 1 : 0;
  // rows rotated in shared memory are rotated by (position - t): q and the output stay unrotated
  p.rel_rope = p.rotate_rows;
  // the chunks of each head group merge inside a cluster when they all run at once
  p.cl_reduce = (p.nch > 1 && p.nch <= 16 && p.items <= sms && p.rel_rope &&
                 attend_max_clusters(p.nch) >= p.items / p.nch) ? 1 : 0;
  p.ncs = p.cl_reduce ? p.nch : 0;
  p.cl_partial = 0;
  if (!p.cl_reduce && p.nch > 1 && p.items <= sms && p.rel_rope) {
    // otherwise: clusters of ncs chunks (the largest size whose clusters all
    // fit at once; the chunk count padded to a multiple with empty chunks)
    // each merge into one partial, and the combine kernel merges those
    for (int ncs = 16; ncs >= 2 && !p.cl_partial; --ncs) {
      const int ncl = (p.nch + ncs - 1) / ncs;
      if (ncl < 2) continue;
      const long long items = units * (long long)ncl * ncs;
      if (items > sms || attend_max_clusters(ncs) < items / ncs) continue;
      p.nch = ncl * ncs;
      p.items = (int)items;
      p.ncs = ncs;
      p.cl_reduce = 1;
      p.cl_partial = 1;
    }
  }
  size_t off = 0;
  const long long parts = p.cl_partial ? (long long)p.items / p.ncs : (long long)p.items;
  if (p.nch > 1 && (!p.cl_reduce || p.cl_partial)) {
    p.off_part_o = off;
    off = align256(off + (size_t)parts * csa::ATT_HG * csa::ATT_D * sizeof(float));
    p.off_part_ml = off;
    off = align256(off + (size_t)parts * csa::ATT_HG * 2 * sizeof(float));
  }
  if (!p.rotate_rows) {
    p.off_rot_ent = off;
    off = align256(off + (size_t)B * N * csa::ATT_D * 2);
    p.off_rot_win = off;
    off = align256(off + (size_t)B * T_win * csa::ATT_D * 2);
  }
  p.bytes = off;
  return p;
}

bool tc_attend_shape(int n_h, int d, int r, int kv_dtype) {
  return d == csa::ATT_D && r == csa::ATT_R && n_h % csa::ATT_HG == 0 &&
         (kv_dtype == CSA_DT_BF16 || kv_dtype == CSA_DT_E4M3_BF16ROPE);
}

template <int NT, int CL, int BITS1, int KEYLO>
csa_status_t launch_topk2_cfg(const csa::Topk2Args& a, int rows, size_t smem, cudaStream_t st,
                              bool pdl) {
  auto kern = csa::topk2_kernel<NT, CL, BITS1, KEYLO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "csa_topk attr");
  if (CL > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_fail(e, "csa_topk cluster attr");
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows * CL);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return cuda_fail(e, "csa_topk launch");
  return CSA_OK;
}

template <int NT, int BITS1, int KEYLO>
csa_status_t launch_topk2_nt(const csa::Topk2Args& a, int CL, int rows, size_t smem, cudaStream_t st,
                             bool pdl) {
  switch (CL) {
    case 1: return launch_topk2_cfg<NT, 1, BITS1, KEYLO>(a, rows, smem, st, pdl);
    case 2: return launch_topk2_cfg<NT, 2, BITS1, KEYLO>(a, rows, smem, st, pdl);
    case 4: return launch_topk2_cfg<NT, 4, BITS1, KEYLO>(a, rows, smem, st, pdl);
    case 8: return launch_topk2_cfg<NT, 8, BITS1, KEYLO>(a, rows, smem, st, pdl);
    default: return launch_topk2_cfg<NT, 16, BITS1, KEYLO>(a, rows, smem, st, pdl);
  }
}

template <int BITS1, int KEYLO>
csa_status_t launch_topk2_keys(const csa::Topk2Args& a, bool wide, int CL, int rows, size_t smem,
                               cudaStream_t st, bool pdl) {
  return wide ? launch_topk2_nt<1024, BITS1, KEYLO>(a, CL, rows, smem, st, pdl)
              : launch_topk2_nt<512, BITS1, KEYLO>(a, CL, rows, smem, st, pdl);
}

// One CTA per row up to 32768 entries, longer rows over a cluster of 8 or 16
// CTAs (rows up to 16 x 32768 entries); 1024 threads per CTA when few CTAs
// run, else 512.  `hist` (optional): per-row histograms of the first
// IDX_HBITS key bits of the visible scores, built by the index kernel.
// A few decode rows of 8K..32K such keys go over a cluster of 16 CTAs of 512
// threads (8 of 1024 when 16 would pass two CTAs per SM): the sweeps are
// barrier-bound, so more, smaller CTAs finish sooner (0.3 us of a 47 us decode
// step at 128K against 8 CTAs of 1024).
csa_status_t launch_topk2(const void* scores, int scores_bf16, const int32_t* q_pos, int32_t* idx,
                          int rows, int Tq, int N, int k, int m, uint32_t* hist, cudaStream_t st) {
  int CL = 1;
  bool few_decode_rows = false;
  if (N > 32768) {
    CL = 8;
    while (CL < 16 && (long long)CL * 32768 < N) CL <<= 1;
  } else if (hist && N > 8192 && (long long)rows * 8 <= 2LL * sm_count()) {
    few_decode_rows = (long long)rows * 16 <= 2LL * sm_count();
    CL = few_decode_rows ? 16 : 8;
  }
  int slice = (N + CL - 1) / CL;
  slice = (slice + 3) & ~3;
  if (slice < 4) slice = 4;
  const int bits1 = hist ? csa::IDX_HBITS : csa::TK2_BITS1;
  const bool merge = CL > 1 && !hist;
  const size_t budget = 200 * 1024;
  const size_t fixed = csa::topk2_smem_bytes(slice, 0, bits1, merge);
  if (fixed > budget) return CSA_ERR_UNSUPPORTED;
  int cand_cap = (int)((budget - fixed) / 4);
  if (cand_cap > slice) cand_cap = slice;
  const size_t smem = csa::topk2_smem_bytes(slice, cand_cap, bits1, merge);
  csa::Topk2Args a{scores, idx, q_pos, Tq, N, k, m, slice, cand_cap, hist};
  const bool wide = !few_decode_rows && (long long)rows * CL <= 2LL * sm_count();
  const bool pdl = kProgrammaticLaunch;
  if (hist) return scores_bf16 ? launch_topk2_keys<csa::IDX_HBITS, 16>(a, wide, CL, rows, smem, st, pdl)
                               : launch_topk2_keys<csa::IDX_HBITS, 0>(a, wide, CL, rows, smem, st, pdl);
  return scores_bf16 ? launch_topk2_keys<csa::TK2_BITS1, 16>(a, wide, CL, rows, smem, st, pdl)
                     : launch_topk2_keys<csa::TK2_BITS1, 0>(a, wide, CL, rows, smem, st, pdl);
}

}  // namespace

extern "C" {

int csa_version(void) { return 1; }

const char* csa_last_cuda_error(void) { return g_cuda_msg; }

const char* csa_status_string(csa_status_t s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case CSA_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA_ERR_CUDA: return "CUDA runtime error";
    case CSA_ERR_TIMEOUT: return "device wait timed out";
    case CSA_ERR_DEVICE: return "device-side fault";
  }
  return "unknown status";
}

csa_status_t csa_device_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(S(stream));
  if (e != cudaSuccess) return cuda_fail(e, "csa_device_error sync");
  unsigned int word = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&word, g_csa_error_word, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e, "csa_device_error read");
  e = cudaMemcpyToSymbol(g_csa_error_word, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e, "csa_device_error clear");
  if (word & ERRBIT_TIMEOUT) return CSA_ERR_TIMEOUT;
  if (word) return CSA_ERR_DEVICE;
  return CSA_OK;
}

// ---------------------------------------------------------------------------
csa_status_t csa_compress_ex(const void* Ca, const void* Cb, const void* Za, const void* Zb,
                             const float* Ba, const float* Bb, void* out, int B, int T, int d,
                             int m, int dtype, const csa_compress_opts_t* opts, void* stream) {
  const int overlap = (Cb != nullptr) ? 1 : 0;
  if ((Cb == nullptr) != (Zb == nullptr)) return CSA_ERR_INVALID_ARG;
  if (B < 0 || T < 0 || d <= 0 || m <= 0 || m > 4096) return CSA_ERR_INVALID_ARG;
  if (dtype != CSA_DT_F32 && dtype != CSA_DT_BF16) return CSA_ERR_UNSUPPORTED;
  const int vec = dtype == CSA_DT_BF16 ? 8 : 4;
  if (d % vec || d / vec > 256) return CSA_ERR_UNSUPPORTED;
  csa_compress_opts_t o;
  memset(&o, 0, sizeof(o));
  if (opts) o = *opts;
  if (o.rms_norm && (!(o.norm_eps >= 0.f) || (o.norm_weight && !aligned(o.norm_weight, 4))))
    return CSA_ERR_INVALID_ARG;
  if (o.rope_dims < 0 || (o.rope_dims & 1) || o.rope_dims > d || o.rope_dims > 128 ||
      (o.rope_dims > 0 && !(o.rope_base > 0.f)))
    return CSA_ERR_INVALID_ARG;
  if (o.rope_dims % vec) return CSA_ERR_UNSUPPORTED;
  RowPages out_pg;
  {
    csa_status_t st = check_pages(&o.out_pages, 0, false, false, &out_pg);
    if (st != CSA_OK) return st;
    if (out_pg.table && (o.out_first < 0 || (o.out_entry0 && !aligned(o.out_entry0, 4))))
      return CSA_ERR_INVALID_ARG;
  }
  if (B == 0 || T / m == 0) return CSA_OK;   // nothing to compress (outputs may be empty)
  if (!Ca || !Za || !out) return CSA_ERR_INVALID_ARG;
  const void* ptrs[] = {Ca, Cb, Za, Zb, out};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return CSA_ERR_INVALID_ARG;
  if ((Ba && !aligned(Ba, 4)) || (Bb && !aligned(Bb, 4))) return CSA_ERR_INVALID_ARG;
  const int N = T / m;
  csa::CompressArgs a;
  memset(&a, 0, sizeof(a));
  a.Ca = Ca; a.Cb = Cb; a.Za = Za; a.Zb = Zb; a.Ba = Ba; a.Bb = Bb; a.out = out;
  a.B = B; a.T = T; a.d = d; a.m = m; a.N = N; a.overlap = overlap;
  a.vecs = d / vec;
  a.rms_norm = o.rms_norm ? 1 : 0;
  a.norm_weight = o.norm_weight;
  a.norm_eps = o.norm_eps;
  a.rope_dims = o.rope_dims;
  if (o.rope_dims > 0) a.rf = make_rope(o.rope_dims, o.rope_base);
  a.out_pg = out_pg;
  a.out_entry0 = out_pg.table ? o.out_entry0 : nullptr;
  a.out_first = out_pg.table ? o.out_first : 0;
  int rows = overlap ? 2 * m : m;
  int groups = 256 / a.vecs;
  if (groups > rows) groups = rows;
  if (groups < 1) groups = 1;
  a.groups = groups;
  dim3 grid(N, B);
  dim3 block(a.vecs * groups);
  size_t smem = ((size_t)groups * a.vecs * 3 * vec + a.vecs) * sizeof(float);
  {
    cudaError_t e = dtype == CSA_DT_BF16
                        ? launch_ex(csa::compress_kernel<__nv_bfloat16>, grid, block, smem, S(stream), 1, a)
                        : launch_ex(csa::compress_kernel<float>, grid, block, smem, S(stream), 1, a);
    if (e != cudaSuccess) return cuda_fail(e, "csa_compress launch");
  }
  return CSA_OK;
}

csa_status_t csa_compress(const void* Ca, const void* Cb, const void* Za, const void* Zb,
                          const float* Ba, const float* Bb, void* out, int B, int T, int d,
                          int m, int dtype, void* stream) {
  return csa_compress_ex(Ca, Cb, Za, Zb, Ba, Bb, out, B, T, d, m, dtype, nullptr, stream);
}

// ---------------------------------------------------------------------------
static csa_status_t index_impl(const void* qI, const void* qI_sf, const float* w, const void* K,
                              const void* K_sf, const csa_pages_t* K_pages, const int32_t* q_pos,
                              void* scores, int score_dtype, int B, int Tq, int N, int H, int c,
                              int m, int dtype, uint32_t* hist, void* stream) {
  if (B < 0 || Tq < 0 || N < 0 || H <= 0 || c <= 0 || m <= 0) return CSA_ERR_INVALID_ARG;
  if (score_dtype != CSA_DT_F32 && score_dtype != CSA_DT_BF16) return CSA_ERR_UNSUPPORTED;
  const int sb = score_dtype == CSA_DT_BF16 ? 1 : 0;
  RowPages kpg;
  csa_status_t pst = check_pages(K_pages, N, false, dtype != CSA_DT_F32, &kpg);
  if (pst != CSA_OK) return pst;
  if (B == 0 || Tq == 0 || N == 0) return CSA_OK;
  if (!qI || !w || !K || !scores) return CSA_ERR_INVALID_ARG;
  if ((q_pos && !aligned(q_pos, 4)) || !aligned(scores, sb ? 2 : 4)) return CSA_ERR_INVALID_ARG;
  if (dtype == CSA_DT_F32) {
    if (c > 256) return CSA_ERR_UNSUPPORTED;
    csa::IndexF32Args a{reinterpret_cast<const float*>(qI), w, reinterpret_cast<const float*>(K),
                        scores, q_pos, sb, kpg, Tq, N, H, c, m};
    dim3 grid((N + 7) / 8, B * Tq);
    cudaError_t e = launch_ex(csa::index_f32_kernel, grid, dim3(256), 0, S(stream), 1, a);
    if (e != cudaSuccess) return cuda_fail(e, "csa_index f32 launch");
    return CSA_OK;
  }
  if (dtype == CSA_DT_BF16) {
    if (!aligned(qI, 16) || !aligned(K, 16) || !aligned(w, 4)) return CSA_ERR_INVALID_ARG;
    if (H == 64 && c == 128)
      return launch_index_tc<64, 128>(qI, w, K, kpg, q_pos, scores, sb, B, Tq, N, m, hist, S(stream));
    if (H == 64 && c == 64)
      return launch_index_tc<64, 64>(qI, w, K, kpg, q_pos, scores, sb, B, Tq, N, m, hist, S(stream));
    if (H == 32 && c == 128)
      return launch_index_tc<32, 128>(qI, w, K, kpg, q_pos, scores, sb, B, Tq, N, m, hist, S(stream));
    if (H == 128 && c == 128)
      return launch_index_tc<128, 128>(qI, w, K, kpg, q_pos, scores, sb, B, Tq, N, m, hist, S(stream));
    return CSA_ERR_UNSUPPORTED;
  }
  if (dtype == CSA_DT_E2M1_BLOCK16) {
    if (!qI_sf || !K_sf) return CSA_ERR_INVALID_ARG;
    if (!aligned(qI, 16) || !aligned(K, 16) || !aligned(qI_sf, 16) || !aligned(K_sf, 16) ||
        !aligned(w, 4))
      return CSA_ERR_INVALID_ARG;
    if (c != csa::FP4_C) return CSA_ERR_UNSUPPORTED;
    if (H == 64)
      return launch_index_fp4<64>(qI, qI_sf, w, K, K_sf, kpg, q_pos, scores, sb, B, Tq, N, m, hist,
                                   S(stream));
    if (H == 32)
      return launch_index_fp4<32>(qI, qI_sf, w, K, K_sf, kpg, q_pos, scores, sb, B, Tq, N, m, hist,
                                   S(stream));
    if (H == 128)
      return launch_index_fp4<128>(qI, qI_sf, w, K, K_sf, kpg, q_pos, scores, sb, B, Tq, N, m, hist,
                                   S(stream));
    return CSA_ERR_UNSUPPORTED;
  }
  return CSA_ERR_UNSUPPORTED;
}

csa_status_t csa_index(const void* qI, const void* qI_sf, const float* w, const void* K,
                       const void* K_sf, const int32_t* q_pos, void* scores, int score_dtype,
                       int B, int Tq, int N, int H, int c, int m, int dtype, void* stream) {
  return index_impl(qI, qI_sf, w, K, K_sf, nullptr, q_pos, scores, score_dtype, B, Tq, N, H, c, m,
                    dtype, nullptr, stream);
}

csa_status_t csa_index_paged(const void* qI, const void* qI_sf, const float* w, const void* K,
                             const void* K_sf, const csa_pages_t* K_pages, const int32_t* q_pos,
                             void* scores, int score_dtype, int B, int Tq, int N, int H, int c,
                             int m, int dtype, void* stream) {
  return index_impl(qI, qI_sf, w, K, K_sf, K_pages, q_pos, scores, score_dtype, B, Tq, N, H, c, m,
                    dtype, nullptr, stream);
}

csa_status_t csa_selftest_wait_timeout(const void* qI, const float* w, const void* K,
                                       const int32_t* q_pos, float* scores, int B, int Tq, int N,
                                       int m, int limit_us, void* stream) {
  if (B <= 0 || Tq <= 0 || N <= 0 || m <= 0 || limit_us < 1 || limit_us > 2000000)
    return CSA_ERR_INVALID_ARG;
  if (!qI || !w || !K || !scores || !aligned(qI, 16) || !aligned(K, 16) || !aligned(w, 4) ||
      !aligned(scores, 4) || (q_pos && !aligned(q_pos, 4)))
    return CSA_ERR_INVALID_ARG;
  const RowPages flat{};
  return launch_index_tc<64, 128>(qI, w, K, flat, q_pos, scores, 0, B, Tq, N, m, nullptr, S(stream),
                                  1000ull * (unsigned long long)limit_us, 1);
}

// ---------------------------------------------------------------------------
static bool index_topk_fused(int B, int Tq, int N, int dtype) {
  return B > 0 && Tq == 1 && N > 0 && N <= 16 * 32768 &&
         (dtype == CSA_DT_BF16 || dtype == CSA_DT_E2M1_BLOCK16);
}

size_t csa_index_topk_workspace_size(int B, int Tq, int N, int dtype) {
  if (!index_topk_fused(B, Tq, N, dtype)) return 0;
  return (size_t)B * Tq * csa::IDX_HBINS * sizeof(uint32_t);
}

csa_status_t csa_index_topk(const void* qI, const void* qI_sf, const float* w, const void* K,
                            const void* K_sf, const int32_t* q_pos, void* scores, int score_dtype,
                            int32_t* idx, int B, int Tq, int N, int H, int c, int m, int k,
                            int dtype, void* ws, size_t ws_bytes, void* stream) {
  return csa_index_topk_paged(qI, qI_sf, w, K, K_sf, nullptr, q_pos, scores, score_dtype, idx, B, Tq,
                              N, H, c, m, k, dtype, ws, ws_bytes, stream);
}

csa_status_t csa_index_topk_paged(const void* qI, const void* qI_sf, const float* w,
                                  const void* K, const void* K_sf, const csa_pages_t* K_pages,
                                  const int32_t* q_pos, void* scores, int score_dtype,
                                  int32_t* idx, int B, int Tq, int N, int H, int c, int m, int k,
                                  int dtype, void* ws, size_t ws_bytes, void* stream) {
  if (k < 1 || k > 4096) return CSA_ERR_INVALID_ARG;
  if (!index_topk_fused(B, Tq, N, dtype)) {
    csa_status_t st = index_impl(qI, qI_sf, w, K, K_sf, K_pages, q_pos, scores, score_dtype, B, Tq,
                                 N, H, c, m, dtype, nullptr, stream);
    if (st != CSA_OK) return st;
    return csa_topk(scores, score_dtype, q_pos, idx, B, Tq, N, k, m, stream);
  }
  if (!idx || !aligned(idx, 4)) return CSA_ERR_INVALID_ARG;
  const size_t need = csa_index_topk_workspace_size(B, Tq, N, dtype);
  if (!ws || ws_bytes < need || !aligned(ws, 16)) return CSA_ERR_WORKSPACE;
  // the histograms start zero (caller's first use) and the selector clears each
  // row's after reading it, so no clearing pass runs here
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws);
  csa_status_t st = index_impl(qI, qI_sf, w, K, K_sf, K_pages, q_pos, scores, score_dtype, B, Tq, N,
                               H, c, m, dtype, hist, stream);
  if (st != CSA_OK) return st;
  return launch_topk2(scores, score_dtype == CSA_DT_BF16, q_pos, idx, B * Tq, Tq, N, k, m, hist,
                      S(stream));
}

// ---------------------------------------------------------------------------
csa_status_t csa_topk(const void* scores, int score_dtype, const int32_t* q_pos, int32_t* idx, int B,
                      int Tq, int N, int k, int m, void* stream) {
  if (B < 0 || Tq < 0 || N < 0 || k < 1 || k > 4096 || m <= 0) return CSA_ERR_INVALID_ARG;
  if (score_dtype != CSA_DT_F32 && score_dtype != CSA_DT_BF16) return CSA_ERR_UNSUPPORTED;
  const int sb = score_dtype == CSA_DT_BF16 ? 1 : 0;
  if (B == 0 || Tq == 0) return CSA_OK;
  if (!idx || (N > 0 && !scores)) return CSA_ERR_INVALID_ARG;
  if (!aligned(scores, sb ? 2 : 4) || !aligned(idx, 4) || (q_pos && !aligned(q_pos, 4)))
    return CSA_ERR_INVALID_ARG;
  const int rows = B * Tq;
  // few long decode rows up to 32768 entries: 8-bit radix passes over a 16-CTA
  // cluster; everything else up to 16 x 32768 entries: the candidate-filtering
  // selector (measured faster there: many short rows, and rows past 32768)
  // (bf16 scores always take the candidate-filtering selector)
  if ((sb || !(N > 8192 && N <= 32768 && rows < 64)) && N <= 16 * 32768)
    return launch_topk2(scores, sb, q_pos, idx, rows, Tq, N, k, m, nullptr, S(stream));
  if (sb) return CSA_ERR_UNSUPPORTED;   // the 8-bit radix selector below reads float32 scores
  // rows longer than 16 slices of 32768 keys: 8-bit radix passes over up to 16 SMs
  int CL = 1;
  if (N > 8192 && rows < 64) CL = rows <= 9 ? 16 : 8;
  int slice = (N + CL - 1) / CL;
  slice = (slice + 3) & ~3;
  const size_t smem = (size_t)slice * sizeof(uint32_t);
  if (smem > 200 * 1024) return CSA_ERR_UNSUPPORTED;
  csa::TopkArgs a{reinterpret_cast<const float*>(scores), idx, q_pos, Tq, N, k, m, slice};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows * CL);
  cfg.blockDim = dim3(csa::TOPK_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = S(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kProgrammaticLaunch ? 2 : 1;
  cudaError_t e;
  switch (CL) {
    case 1:
      e = cudaFuncSetAttribute(csa::topk_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return cuda_fail(e, "csa_topk attr");
      e = cudaLaunchKernelEx(&cfg, csa::topk_kernel<1>, a);
      break;
    case 8:
      e = cudaFuncSetAttribute(csa::topk_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return cuda_fail(e, "csa_topk attr");
      e = cudaLaunchKernelEx(&cfg, csa::topk_kernel<8>, a);
      break;
    default:
      e = cudaFuncSetAttribute(csa::topk_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return cuda_fail(e, "csa_topk attr");
      e = cudaFuncSetAttribute(csa::topk_kernel<16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return cuda_fail(e, "csa_topk attr");
      e = cudaLaunchKernelEx(&cfg, csa::topk_kernel<16>, a);
      break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "csa_topk launch");
  return CSA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// csa_attend / hca_attend: arguments, host-side checks, plan and launches.
namespace {

struct AttendCall {
  const void* q;
  csa_kv_t ent, win;
  const int32_t* idx;
  const int32_t* q_pos;
  const int32_t* win_base;
  const float* sink;
  void* out;
  int B, Tq, N, k, T_win, n_h, d, r, m, n_win;
  float rope_base;
  int dense;
};

// Every host-side check of an attention call (sizes, null and misaligned
// pointers, supported shapes).  Returns CSA_OK with *plan set for a launch, or
// CSA_OK with *empty = true when there is nothing to do.
csa_status_t attend_validate(const AttendCall& c, AttPlan* plan, bool* empty) {
  *empty = false;
  if (c.B < 0 || c.Tq < 0 || c.N < 0 || c.T_win < 0 || c.n_h <= 0 || c.d <= 0 || c.r < 0 ||
      c.r > c.d || (c.r & 1) || c.r > 128 || c.m <= 0 || c.n_win <= 0 || !(c.rope_base > 0.f))
    return CSA_ERR_INVALID_ARG;
  if (!c.dense && (c.k < 1 || c.k > 4096)) return CSA_ERR_INVALID_ARG;
  if (c.N > 0 && !c.ent.data) return CSA_ERR_INVALID_ARG;
  if ((c.ent.flags & ~CSA_KV_ROTATED) || (c.win.flags & ~CSA_KV_ROTATED)) return CSA_ERR_INVALID_ARG;
  if (c.win.flags) return CSA_ERR_UNSUPPORTED;   // window rows are stored unrotated
  {
    RowPages pg;
    csa_status_t st = check_pages(&c.ent.pages, c.N, false, false, &pg);
    if (st == CSA_OK) st = check_pages(&c.win.pages, c.T_win, true, false, &pg);
    if (st != CSA_OK) return st;
  }
  if (c.B == 0 || c.Tq == 0) {
    *empty = true;
    return CSA_OK;
  }
  if (!c.q || !c.sink || !c.out || (c.T_win > 0 && !c.win.data)) return CSA_ERR_INVALID_ARG;
  if (!c.dense && !c.idx) return CSA_ERR_INVALID_ARG;
  if ((c.q_pos && !aligned(c.q_pos, 4)) || (c.win_base && !aligned(c.win_base, 4)) ||
      (c.idx && !aligned(c.idx, 4)))
    return CSA_ERR_INVALID_ARG;
  if (c.ent.dtype == CSA_DT_F32 && c.win.dtype == CSA_DT_F32) {
    if (c.d > 512 || (size_t)c.n_h * c.d > 16384) return CSA_ERR_UNSUPPORTED;
    memset(plan, 0, sizeof(*plan));
    return CSA_OK;
  }
  if (!tc_attend_shape(c.n_h, c.d, c.r, c.ent.dtype) || c.ent.dtype != c.win.dtype)
    return CSA_ERR_UNSUPPORTED;
  const int mixed = c.ent.dtype == CSA_DT_E4M3_BF16ROPE;
  if (!aligned(c.q, 16) || !aligned(c.out, 16) || (c.T_win > 0 && !aligned(c.win.data, 16)) ||
      (c.N > 0 && !aligned(c.ent.data, 16)))
    return CSA_ERR_INVALID_ARG;
  if (mixed && ((c.T_win > 0 && (!c.win.scale || !c.win.rope || !aligned(c.win.rope, 16))) ||
                (c.N > 0 && (!c.ent.scale || !c.ent.rope || !aligned(c.ent.rope, 16)))))
    return CSA_ERR_INVALID_ARG;
  if ((long long)c.B * c.N >= 0x7fffffffLL || (long long)c.B * c.T_win >= 0x7fffffffLL ||
      (long long)c.B * c.Tq * c.n_h >= 0x7fffffffLL)
    return CSA_ERR_UNSUPPORTED;
  *plan = plan_attend(c.B, c.Tq, c.N, c.dense ? 0 : c.k, c.T_win, c.n_h, c.n_win, c.dense, mixed);
  return CSA_OK;
}

// The launches of a validated call; ws holds at least plan.bytes (256-byte aligned).
csa_status_t attend_launch(const AttendCall& c, const AttPlan& p, void* ws, void* stream) {
  const RopeFreqs rf = make_rope(c.r, c.rope_base);
  cudaStream_t st = S(stream);
  RowPages ent_pg, win_pg;      // checked in attend_validate
  check_pages(&c.ent.pages, c.N, false, false, &ent_pg);
  check_pages(&c.win.pages, c.T_win, true, false, &win_pg);
  if (c.ent.dtype == CSA_DT_F32 && c.win.dtype == CSA_DT_F32) {
    csa::AttendF32Args a;
    memset(&a, 0, sizeof(a));
    a.q = reinterpret_cast<const float*>(c.q);
    a.ent = reinterpret_cast<const float*>(c.ent.data);
    a.idx = c.dense ? nullptr : c.idx;
    a.win = reinterpret_cast<const float*>(c.win.data);
    a.sink = c.sink;
    a.out = reinterpret_cast<float*>(c.out);
    a.q_pos = c.q_pos; a.win_base = c.win_base;
    a.Tq = c.Tq; a.N = c.N; a.k = c.dense ? 0 : c.k; a.T_win = c.T_win;
    a.n_h = c.n_h; a.d = c.d; a.r = c.r; a.m = c.m; a.n_win = c.n_win;
    a.dense = c.dense;
    a.ent_rotated = (c.ent.flags & CSA_KV_ROTATED) ? 1 : 0;
    a.ent_pg = ent_pg; a.win_pg = win_pg;
    a.inv_sqrt_d = (float)(1.0 / std::sqrt((double)c.d));
    a.rf = rf;
    const size_t smem = ((size_t)2 * c.n_h * c.d + c.d + 5 * c.n_h) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(csa::attend_f32_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "csa_attend f32 attr");
    e = launch_ex(csa::attend_f32_kernel, dim3(c.B * c.Tq), dim3(csa::ATT_F32_THREADS), smem, st, 1, a);
    if (e != cudaSuccess) return cuda_fail(e, "csa_attend f32 launch");
    return CSA_OK;
  }
  const int mixed = c.ent.dtype == CSA_DT_E4M3_BF16ROPE;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  csa::AttendTcArgs a;
  memset(&a, 0, sizeof(a));
  a.q = reinterpret_cast<const __nv_bfloat16*>(c.q);
  a.ent = c.ent.data; a.ent_scale = c.ent.scale;
  a.ent_rope = reinterpret_cast<const __nv_bfloat16*>(c.ent.rope);
  a.win = c.win.data; a.win_scale = c.win.scale;
  a.win_rope = reinterpret_cast<const __nv_bfloat16*>(c.win.rope);
  a.idx = c.dense ? nullptr : c.idx;
  a.q_pos = c.q_pos; a.win_base = c.win_base;
  a.sink = c.sink;
  a.out = reinterpret_cast<__nv_bfloat16*>(c.out);
  a.B = c.B; a.Tq = c.Tq; a.N = c.N; a.k = c.dense ? 0 : c.k; a.T_win = c.T_win;
  a.n_h = c.n_h; a.m = c.m; a.n_win = c.n_win;
  a.HG = p.HG; a.nch = p.nch; a.chunk_rows = p.chunk_rows; a.items = p.items;
  a.rotate_rows = p.rotate_rows; a.kv_mixed = mixed;
  a.cl_reduce = p.cl_reduce;
  a.ncs = p.ncs;
  a.cl_partial = p.cl_partial;
  a.rel_rope = p.rel_rope;
  a.ent_rotated = (c.ent.flags & CSA_KV_ROTATED) ? 1 : 0;
  a.ent_pg = ent_pg; a.win_pg = win_pg;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c.d));
  a.rf = rf;
  if (!p.rotate_rows) {
    // rotate the RoPE dims of every stored row once
    csa::RotateArgs ra;
    memset(&ra, 0, sizeof(ra));
    ra.rf = rf;
    if (c.N > 0 && !a.ent_rotated) {
      ra.src = reinterpret_cast<const __nv_bfloat16*>(c.ent.data);
      ra.dst = reinterpret_cast<__nv_bfloat16*>(wsb + p.off_rot_ent);
      ra.rows = (long long)c.B * c.N; ra.rows_per_b = c.N; ra.m = c.m; ra.base = nullptr;
      ra.pg = ent_pg;
      cudaError_t e = launch_ex(csa::rope_rotate_rows_kernel, dim3((unsigned)((ra.rows * 64 + 255) / 256)),
                                dim3(256), 0, st, 1, ra);
      if (e != cudaSuccess) return cuda_fail(e, "csa_attend rotate entries");
      a.ent = ra.dst;
      memset(&a.ent_pg, 0, sizeof(a.ent_pg));     // the rotated copy is flat
    }
    if (c.T_win > 0) {
      ra.src = reinterpret_cast<const __nv_bfloat16*>(c.win.data);
      ra.dst = reinterpret_cast<__nv_bfloat16*>(wsb + p.off_rot_win);
      ra.rows = (long long)c.B * c.T_win; ra.rows_per_b = c.T_win; ra.m = 0; ra.base = c.win_base;
      ra.pg = win_pg;
      cudaError_t e = launch_ex(csa::rope_rotate_rows_kernel, dim3((unsigned)((ra.rows * 64 + 255) / 256)),
                                dim3(256), 0, st, 1, ra);
      if (e != cudaSuccess) return cuda_fail(e, "csa_attend rotate window");
      a.win = ra.dst;
      memset(&a.win_pg, 0, sizeof(a.win_pg));     // flat, token order from win_base
    }
  }
  if (p.nch > 1 && (!p.cl_reduce || p.cl_partial)) {
    a.part_o = reinterpret_cast<float*>(wsb + p.off_part_o);
    a.part_ml = reinterpret_cast<float*>(wsb + p.off_part_ml);
  }
  CUtensorMap tmq;
  memset(&tmq, 0, sizeof(tmq));
  if (!tmap_bf16_3d(&tmq, c.q, csa::ATT_D, (uint64_t)c.B * c.Tq * c.n_h, 1, (uint64_t)csa::ATT_D * 2,
                    (uint64_t)c.B * c.Tq * c.n_h * csa::ATT_D * 2, 64, csa::ATT_HG))
    return CSA_ERR_UNSUPPORTED;
  const int smem = csa::AttSmem::BYTES;
  cudaError_t e = cudaFuncSetAttribute(csa::attend_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "csa_attend tc attr");
  const int sms = sm_count();
  const int grid = p.items < sms ? p.items : sms;
  if (p.cl_reduce && p.ncs > 8) {
    e = cudaFuncSetAttribute(csa::attend_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_fail(e, "csa_attend cluster attr");
  }
  const bool pdl = p.items <= (long long)kProgrammaticAttendItems * sms;
  e = launch_ex_pdl(csa::attend_tc_kernel, dim3(grid), dim3(csa::ATT_THREADS), smem, st,
                    p.cl_reduce ? p.ncs : 1, pdl, tmq, a);
  if (e != cudaSuccess) return cuda_fail(e, "csa_attend tc launch");
  if (p.nch > 1 && (!p.cl_reduce || p.cl_partial)) {
    csa::CombineArgs ca;
    memset(&ca, 0, sizeof(ca));
    ca.part_o = a.part_o; ca.part_ml = a.part_ml; ca.sink = c.sink; ca.out = a.out;
    ca.q_pos = c.q_pos;
    ca.Tq = c.Tq; ca.n_h = c.n_h; ca.HG = p.HG; ca.rf = rf;
    ca.nch = p.cl_partial ? p.nch / p.ncs : p.nch;     // partials per (query row, head group)
    ca.rel_rope = p.rel_rope;
    const size_t cmb_smem = (size_t)ca.nch * csa::ATT_HG * 2 * sizeof(float);
    if (cmb_smem > 48 * 1024) {
      e = cudaFuncSetAttribute(csa::attend_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)cmb_smem);
      if (e != cudaSuccess) return cuda_fail(e, "csa_attend combine attr");
    }
    e = launch_ex(csa::attend_combine_kernel,
                  dim3((unsigned)((size_t)c.B * c.Tq * p.HG * (csa::ATT_D / csa::CMB_DIMS))),
                  dim3(csa::CMB_THREADS), cmb_smem, st, 1, ca);
    if (e != cudaSuccess) return cuda_fail(e, "csa_attend combine launch");
  }
  return CSA_OK;
}

csa_status_t attend_with_workspace(const AttendCall& c, void* ws, size_t ws_bytes, void* stream) {
  AttPlan p;
  bool empty = false;
  csa_status_t st = attend_validate(c, &p, &empty);
  if (st != CSA_OK || empty) return st;
  if (p.bytes > 0 && (!ws || ws_bytes < p.bytes || !aligned(ws, 256))) return CSA_ERR_WORKSPACE;
  return attend_launch(c, p, ws, stream);
}

}  // namespace

extern "C" {

csa_status_t csa_attend(const void* q, csa_kv_t entries, const int32_t* idx, csa_kv_t win,
                        const int32_t* q_pos, const int32_t* win_base, const float* sink,
                        void* out, int B, int Tq, int N, int k, int T_win, int n_h, int d, int r,
                        int m, int n_win, float rope_base, void* ws, size_t ws_bytes,
                        void* stream) {
  const AttendCall c{q, entries, win, idx, q_pos, win_base, sink, out, B, Tq, N, k, T_win,
                     n_h, d, r, m, n_win, rope_base, 0};
  return attend_with_workspace(c, ws, ws_bytes, stream);
}

csa_status_t hca_attend(const void* q, csa_kv_t entries, csa_kv_t win, const int32_t* q_pos,
                        const int32_t* win_base, const float* sink, void* out, int B, int Tq,
                        int N, int T_win, int n_h, int d, int r, int m, int n_win,
                        float rope_base, void* ws, size_t ws_bytes, void* stream) {
  const AttendCall c{q, entries, win, nullptr, q_pos, win_base, sink, out, B, Tq, N, 0, T_win,
                     n_h, d, r, m, n_win, rope_base, 1};
  return attend_with_workspace(c, ws, ws_bytes, stream);
}

size_t csa_attend_workspace_size(int B, int Tq, int N, int k, int T_win, int n_h, int d, int r,
                                 int m, int n_win, int q_dtype, int kv_dtype, int is_hca) {
  (void)q_dtype;
  if (B <= 0 || Tq <= 0 || n_h <= 0 || m <= 0 || N < 0 || T_win < 0 || n_win <= 0) return 0;
  if (!tc_attend_shape(n_h, d, r, kv_dtype)) return 0;
  return plan_attend(B, Tq, N, is_hca ? 0 : k, T_win, n_h, n_win, is_hca ? 1 : 0,
                     kv_dtype == CSA_DT_E4M3_BF16ROPE ? 1 : 0).bytes;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// csa_decode_step_host: one decode step from host buffers.  Scratch layout:
// staged inputs, float32 scores, indices, device output, the top-k histograms
// (zero between calls), the attention's scratch; every part 256-byte aligned.
struct StepLayout {
  size_t q, qi, qisf, w, qpos, wb, scores, idx, out, hist, nhist, att, natt, bytes;
};

static bool step_layout(int B, int N, int H, int c, int k, int T_win, int n_h, int d, int r, int m,
                        int n_win, int dtype, int kv_dtype, StepLayout* L) {
  if (B <= 0 || N <= 0 || H <= 0 || c <= 0 || (c & 15) || k < 1 || k > 4096 || T_win < 0 ||
      n_h <= 0 || d <= 0 || m <= 0 || n_win <= 0)
    return false;
  if (dtype != CSA_DT_BF16 && dtype != CSA_DT_E2M1_BLOCK16) return false;
  if (kv_dtype != CSA_DT_BF16 && kv_dtype != CSA_DT_E4M3_BF16ROPE) return false;
  const bool fp4 = dtype == CSA_DT_E2M1_BLOCK16;
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t o = off;
    off = align256(off + n);
    return o;
  };
  L->q = take((size_t)B * n_h * d * 2);
  L->qi = take((size_t)B * H * (fp4 ? c / 2 : c * 2));
  L->qisf = take(fp4 ? (size_t)B * H * (c / 16) : 0);
  L->w = take((size_t)B * H * 4);
  L->qpos = take((size_t)B * 4);
  L->wb = take((size_t)B * 4);
  L->scores = take((size_t)B * N * 4);
  L->idx = take((size_t)B * k * 4);
  L->out = take((size_t)B * n_h * d * 2);
  L->nhist = csa_index_topk_workspace_size(B, 1, N, dtype);
  L->hist = take(L->nhist);
  L->natt = csa_attend_workspace_size(B, 1, N, k, T_win, n_h, d, r, m, n_win, CSA_DT_BF16, kv_dtype, 0);
  L->att = take(L->natt);
  L->bytes = off;
  return true;
}

size_t csa_decode_step_workspace_size(int B, int N, int H, int c, int k, int T_win, int n_h, int d,
                                      int r, int m, int n_win, int dtype, int kv_dtype) {
  StepLayout L;
  return step_layout(B, N, H, c, k, T_win, n_h, d, r, m, n_win, dtype, kv_dtype, &L) ? L.bytes : 0;
}

csa_status_t csa_decode_step_host(const void* q_h, const void* qI_h, const void* qI_sf_h,
                                  const float* w_h, const int32_t* q_pos_h,
                                  const int32_t* win_base_h, const void* K, const void* K_sf,
                                  const csa_pages_t* K_pages, csa_kv_t entries, csa_kv_t win,
                                  const float* sink, void* out_h, int B, int N, int H, int c, int k,
                                  int T_win, int n_h, int d, int r, int m, int n_win, int dtype,
                                  float rope_base, void* ws, size_t ws_bytes, void* stream) {
  StepLayout L;
  if (!step_layout(B, N, H, c, k, T_win, n_h, d, r, m, n_win, dtype, entries.dtype, &L))
    return CSA_ERR_INVALID_ARG;
  const bool fp4 = dtype == CSA_DT_E2M1_BLOCK16;
  if (!q_h || !qI_h || !w_h || !q_pos_h || !out_h || !sink || !K || (fp4 && (!qI_sf_h || !K_sf)))
    return CSA_ERR_INVALID_ARG;
  if (!ws || ws_bytes < L.bytes || !aligned(ws, 256)) return CSA_ERR_WORKSPACE;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  cudaStream_t st = S(stream);
  // the step's new inputs, host -> device
  const struct { size_t off; const void* src; size_t n; } in[] = {
      {L.q, q_h, (size_t)B * n_h * d * 2},
      {L.qi, qI_h, (size_t)B * H * (fp4 ? c / 2 : c * 2)},
      {L.qisf, fp4 ? qI_sf_h : nullptr, fp4 ? (size_t)B * H * (c / 16) : 0},
      {L.w, w_h, (size_t)B * H * 4},
      {L.qpos, q_pos_h, (size_t)B * 4},
      {L.wb, win_base_h, win_base_h ? (size_t)B * 4 : 0},
  };
  for (const auto& e : in) {
    if (!e.n) continue;
    const cudaError_t ce = cudaMemcpyAsync(wsb + e.off, e.src, e.n, cudaMemcpyHostToDevice, st);
    if (ce != cudaSuccess) return cuda_fail(ce, "csa_decode_step_host copy in");
  }
  const int32_t* qpos = reinterpret_cast<const int32_t*>(wsb + L.qpos);
  int32_t* idx = reinterpret_cast<int32_t*>(wsb + L.idx);
  csa_status_t s = csa_index_topk_paged(
      wsb + L.qi, fp4 ? wsb + L.qisf : nullptr, reinterpret_cast<const float*>(wsb + L.w), K,
      fp4 ? K_sf : nullptr, K_pages, qpos, wsb + L.scores, CSA_DT_F32, idx, B, 1, N, H, c, m, k, dtype,
      L.nhist ? wsb + L.hist : nullptr, L.nhist, stream);
  if (s != CSA_OK) return s;
  s = csa_attend(wsb + L.q, entries, idx, win, qpos,
                 win_base_h ? reinterpret_cast<const int32_t*>(wsb + L.wb) : nullptr, sink, wsb + L.out,
                 B, 1, N, k, T_win, n_h, d, r, m, n_win, rope_base, L.natt ? wsb + L.att : nullptr,
                 L.natt, stream);
  if (s != CSA_OK) return s;
  const cudaError_t ce =
      cudaMemcpyAsync(out_h, wsb + L.out, (size_t)B * n_h * d * 2, cudaMemcpyDeviceToHost, st);
  if (ce != cudaSuccess) return cuda_fail(ce, "csa_decode_step_host copy out");
  return CSA_OK;
}

// ---------------------------------------------------------------------------
// csa_attend_noalloc: csa_attend for callers that cannot allocate device
// memory.  Its scratch is one fixed array in this library's device image.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_attend_noalloc_scratch[CSA_NOALLOC_SCRATCH_BYTES];

namespace {

typedef CUresult (*PFN_ctx_get_current)(CUcontext*);
typedef CUresult (*PFN_ctx_get_id)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (driver calls reached
// through the runtime's entry-point query, so the library needs no -lcuda).
// Ids are never reused within a process, unlike context handles, so a context
// made after cudaDeviceReset never matches an address cached for the old one.
bool current_context_id(unsigned long long* id) {
  static PFN_ctx_get_current get_cur = nullptr;
  static PFN_ctx_get_id get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_ctx_get_current>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_ctx_get_id>(p);
  });
  CUcontext ctx = nullptr;
  if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

constexpr int kNoallocCacheSlots = 64;
std::mutex g_noalloc_mu;
unsigned long long g_noalloc_ctx[kNoallocCacheSlots] = {};
void* g_noalloc_ptr[kNoallocCacheSlots] = {};
int g_noalloc_next = 0;

// Device address of the scratch array in the calling thread's current context.
// The array's name in host code is only a host-side handle, and each context
// that loads this library has its own copy at its own address, so the address
// is looked up (cudaGetSymbolAddress) once per context and cached under the
// context's unique id.
csa_status_t noalloc_scratch(void** out) {
  unsigned long long id = 0;
  if (current_context_id(&id)) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    for (int i = 0; i < kNoallocCacheSlots; ++i)
      if (g_noalloc_ptr[i] && g_noalloc_ctx[i] == id) {
        *out = g_noalloc_ptr[i];
        return CSA_OK;
      }
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_attend_noalloc_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "csa_attend_noalloc scratch address");
  // the lookup made the device's context current if none was: cache under its id
  if (current_context_id(&id)) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    g_noalloc_ctx[g_noalloc_next] = id;
    g_noalloc_ptr[g_noalloc_next] = p;
    g_noalloc_next = (g_noalloc_next + 1) % kNoallocCacheSlots;
  }
  *out = p;
  return CSA_OK;
}

}  // namespace

extern "C" csa_status_t csa_attend_noalloc(const void* q, csa_kv_t entries, const int32_t* idx,
                                           csa_kv_t win, const int32_t* q_pos,
                                           const int32_t* win_base, const float* sink, void* out,
                                           int B, int Tq, int N, int k, int T_win, int n_h, int d,
                                           int r, int m, int n_win, float rope_base,
                                           void* stream) {
  const AttendCall c{q, entries, win, idx, q_pos, win_base, sink, out, B, Tq, N, k, T_win,
                     n_h, d, r, m, n_win, rope_base, 0};
  AttPlan p;
  bool empty = false;
  csa_status_t st = attend_validate(c, &p, &empty);   // argument errors come first
  if (st != CSA_OK || empty) return st;
  if (p.bytes > CSA_NOALLOC_SCRATCH_BYTES) {
    snprintf(g_cuda_msg, sizeof(g_cuda_msg),
             "csa_attend_noalloc: these sizes need %zu scratch bytes, above the fixed %zu", p.bytes,
             (size_t)CSA_NOALLOC_SCRATCH_BYTES);
    return CSA_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  if (p.bytes > 0) {
    st = noalloc_scratch(&ws);
    if (st != CSA_OK) return st;
  }
  return attend_launch(c, p, ws, stream);
}

// ---------------------------------------------------------------------------
// csa_grouped_proj: the grouped output projection (and, with G = 1, the final
// projection to the model width) as one tcgen05 GEMM per call.
extern "C" csa_status_t csa_grouped_proj(const void* A, int64_t lda, const void* W, void* C,
                                         int64_t ldc, int M, int N, int K, int G, void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || G <= 0) return CSA_ERR_INVALID_ARG;
  if (lda < (int64_t)G * K || ldc < (int64_t)G * N) return CSA_ERR_INVALID_ARG;
  if (M == 0) return CSA_OK;
  if (!A || !W || !C) return CSA_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(W, 16) || !aligned(C, 16)) return CSA_ERR_INVALID_ARG;
  // TMA strides are multiples of 16 bytes; the vector stores need 8-element rows
  if (K % 8 || lda % 8 || ldc % 8 || N % 8) return CSA_ERR_UNSUPPORTED;
  csa::GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.C = reinterpret_cast<__nv_bfloat16*>(C);
  a.ldc = ldc;
  a.M = M; a.N = N; a.K = K; a.G = G;
  a.MT = (M + csa::GEMM_BM - 1) / csa::GEMM_BM;
  a.NT = (N + csa::GEMM_BN - 1) / csa::GEMM_BN;
  a.tiles = (long long)G * a.MT * a.NT;
  CUtensorMap tmA, tmW;
  const uint64_t dA[3] = {(uint64_t)K, (uint64_t)G, (uint64_t)M};
  const uint64_t sA[2] = {(uint64_t)K * 2, (uint64_t)lda * 2};
  const uint32_t bA[3] = {(uint32_t)csa::GEMM_BK, 1, (uint32_t)csa::GEMM_BM};
  const uint64_t dW[3] = {(uint64_t)K, (uint64_t)N, (uint64_t)G};
  const uint64_t sW[2] = {(uint64_t)K * 2, (uint64_t)N * K * 2};
  const uint32_t bW[3] = {(uint32_t)csa::GEMM_BK, (uint32_t)csa::GEMM_BN, 1};
  if (!tmap_bf16_3d_box(&tmA, A, dA, sA, bA) || !tmap_bf16_3d_box(&tmW, W, dW, sW, bW))
    return CSA_ERR_UNSUPPORTED;
  const int smem = csa::GemmSmem::BYTES;
  cudaError_t e = cudaFuncSetAttribute(csa::gemm_grouped_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "csa_grouped_proj attr");
  const int sms = sm_count();
  const int grid = a.tiles < sms ? (int)a.tiles : sms;
  e = launch_ex(csa::gemm_grouped_kernel, dim3(grid), dim3(csa::GEMM_THREADS), smem, S(stream), 1,
                tmA, tmW, a);
  if (e != cudaSuccess) return cuda_fail(e, "csa_grouped_proj launch");
  return CSA_OK;
}

// ---------------------------------------------------------------------------
// Block pool: the free physical blocks of a paged cache, as a stack of ids
// (host memory only).  `used` marks allocated ids so that a release of an id
// that is free, out of range or repeated is refused whole.
struct csa_block_pool {
  std::vector<int32_t> free_ids;     // top of the stack = next id handed out
  std::vector<uint8_t> used;
};

extern "C" csa_block_pool_t* csa_block_pool_create(int32_t num_blocks) {
  if (num_blocks < 1 || num_blocks > (1 << 30)) return nullptr;
  csa_block_pool_t* p = new (std::nothrow) csa_block_pool_t();
  if (!p) return nullptr;
  try {
    p->used.assign((size_t)num_blocks, 0);
    p->free_ids.resize((size_t)num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) p->free_ids[(size_t)i] = num_blocks - 1 - i;
  } catch (...) {
    delete p;
    return nullptr;
  }
  return p;
}

extern "C" void csa_block_pool_destroy(csa_block_pool_t* pool) { delete pool; }

extern "C" int32_t csa_block_pool_free_count(const csa_block_pool_t* pool) {
  return pool ? (int32_t)pool->free_ids.size() : 0;
}

extern "C" csa_status_t csa_block_pool_alloc(csa_block_pool_t* pool, int32_t n, int32_t* ids) {
  if (!pool || n < 0 || (n > 0 && !ids)) return CSA_ERR_INVALID_ARG;
  if ((size_t)n > pool->free_ids.size()) return CSA_ERR_WORKSPACE;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = pool->free_ids.back();
    pool->free_ids.pop_back();
    pool->used[(size_t)id] = 1;
    ids[i] = id;
  }
  return CSA_OK;
}

extern "C" csa_status_t csa_block_pool_release(csa_block_pool_t* pool, int32_t n,
                                               const int32_t* ids) {
  if (!pool || n < 0 || (n > 0 && !ids)) return CSA_ERR_INVALID_ARG;
  const size_t nb = pool->used.size();
  int32_t i = 0;
  for (; i < n; ++i) {                 // check every id first (2 marks a repeat)
    const int32_t id = ids[i];
    if (id < 0 || (size_t)id >= nb || pool->used[(size_t)id] != 1) break;
    pool->used[(size_t)id] = 2;
  }
  if (i < n) {                         // refused: undo the marks
    for (int32_t j = 0; j < i; ++j) pool->used[(size_t)ids[j]] = 1;
    return CSA_ERR_INVALID_ARG;
  }
  for (int32_t j = n - 1; j >= 0; --j) {
    pool->used[(size_t)ids[j]] = 0;
    pool->free_ids.push_back(ids[j]);
  }
  return CSA_OK;
}

#ifdef CSA_TRACE
// Phase marks of the traced library variant: copies n <= CSA_TRACE_CTAS *
// CSA_TRACE_SLOTS marks (row = CTA, column = slot) to host memory and clears them.
extern "C" int csa_trace_read(long long* host, int n) {
  const int cap = csa::CSA_TRACE_CTAS * csa::CSA_TRACE_SLOTS;
  if (!host || n < 0) return -1;
  if (n > cap) n = cap;
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(host, csa::g_csa_trace, (size_t)n * sizeof(long long)) != cudaSuccess)
    return -1;
  static long long zeros[csa::CSA_TRACE_CTAS * csa::CSA_TRACE_SLOTS];
  if (cudaMemcpyToSymbol(csa::g_csa_trace, zeros, sizeof(zeros)) != cudaSuccess) return -1;
  return n;
}

// Which tile of each CTA the attention kernel's per-tile marks describe (0 = first).
extern "C" int csa_trace_set_tile(int tile) {
  return cudaMemcpyToSymbol(csa::g_csa_trace_tile, &tile, sizeof(tile)) == cudaSuccess ? 0 : -1;
}
#endif
