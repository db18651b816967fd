// C ABI of the CSA / HCA forward kernels (declared in include/csa.h).
//
// One translation unit: the kernels live in the included .cuh files so that
// they share the device error word without relocatable device code.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/csa.h"
#include "common.cuh"
#include "compress.cuh"
#include "topk.cuh"
#include "topk2.cuh"
#include "simt_f32.cuh"
#include "index_tc.cuh"
#include "index_fp4.cuh"
#include "attend_tc.cuh"

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


// Programmatic stream serialisation would let a kernel start while the previous
// kernel in the stream finishes (every kernel here waits on the grid dependency
// before its first global memory access, so either setting is correct).  Off:
// measured in CUDA-graph replay of the decode and prefill steps, the early-
// launched grids made each step slower (decode 128K: 69 vs 59 us per step).
constexpr bool kProgrammaticLaunch = false;

// Launch with an optional cluster size (and programmatic serialisation when on).
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (kProgrammaticLaunch) {
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

template <int H>
csa_status_t launch_index_fp4(const void* qI, const void* qI_sf, const float* w, const void* K,
                              const void* K_sf, float* scores, int B, int Tq, int N, int m,
                              int q_pos0, uint32_t* hist, cudaStream_t stream) {
  csa::IndexFp4Args fa;
  memset(&fa, 0, sizeof(fa));
  csa::IndexTcArgs& a = fa.t;
  a.w = w; a.scores = scores; a.B = B; a.Tq = Tq; a.N = N; a.m = m; a.q_pos0 = q_pos0;
  csa_status_t st = plan_index(a, 128 / H, B, Tq, N);
  if (st != CSA_OK) return st;
  if ((long long)B * N >= 0x7fffffffLL || (long long)B * Tq * H >= 0x7fffffffLL)
    return CSA_ERR_UNSUPPORTED;
  fa.sf_rows = (long long)B * N;
  a.hist = a.QT == 1 ? hist : nullptr;
  const int nqh = a.QT * H;
  a.tmem_cols = 512;
  // accumulator buffers in columns [0, 256), scale factors above; the two
  // epilogue groups take alternate buffers
  a.nbuf = 4 * nqh <= 256 ? 4 : 2;
  CUtensorMap tmK, tmq, tmKs, tmqs;
  if (!tmap_u8_3d_sw64(&tmK, K, csa::FP4_ROWB, N, B, csa::FP4_ROWB, (uint64_t)N * csa::FP4_ROWB,
                       csa::IDX_TILE) ||
      !tmap_u8_3d_sw64(&tmq, qI, csa::FP4_ROWB, (uint64_t)Tq * H, B, csa::FP4_ROWB,
                       (uint64_t)Tq * H * csa::FP4_ROWB, nqh) ||
      !tmap_u64_1d(&tmKs, K_sf, (uint64_t)B * N, csa::FP4_SF_BOX) ||
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
csa_status_t launch_index_tc(const void* qI, const float* w, const void* K, float* scores, int B,
                             int Tq, int N, int m, int q_pos0, uint32_t* hist, cudaStream_t stream) {
  csa::IndexTcArgs a;
  a.w = w; a.scores = scores; a.B = B; a.Tq = Tq; a.N = N; a.m = m; a.q_pos0 = q_pos0;
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
  if (!tmap_bf16_3d(&tmK, K, C, N, B, (uint64_t)C * 2, (uint64_t)N * C * 2, 64, csa::IDX_TILE) ||
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

AttPlan plan_attend(int B, int Tq, int N, int k, int T_win, int n_h, int m, int n_win, int q_pos0,
                    int dense, int kv_mixed) {
  AttPlan p;
  memset(&p, 0, sizeof(p));
  p.HG = n_h / csa::ATT_HG;
  const long long t_last = (long long)q_pos0 + Tq - 1;
  long long vis = (t_last + 1) / m;
  if (vis > N) vis = N;
  const long long nsel = dense ? vis : (vis < k ? vis : k);
  const long long win = t_last + 1 < n_win ? t_last + 1 : n_win;
  const long long rows_max = nsel + win;
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
  size_t off = 0;
  if (p.nch > 1 && !p.cl_reduce) {
    p.off_part_o = off;
    off = align256(off + (size_t)p.items * csa::ATT_HG * csa::ATT_D * sizeof(float));
    p.off_part_ml = off;
    off = align256(off + (size_t)p.items * csa::ATT_HG * 2 * sizeof(float));
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

template <int NT, int CL, int BITS1>
csa_status_t launch_topk2_cfg(const csa::Topk2Args& a, int rows, size_t smem, cudaStream_t st) {
  auto kern = csa::topk2_kernel<NT, CL, BITS1>;
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
  cfg.numAttrs = kProgrammaticLaunch ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return cuda_fail(e, "csa_topk launch");
  return CSA_OK;
}

template <int NT, int BITS1>
csa_status_t launch_topk2_nt(const csa::Topk2Args& a, int CL, int rows, size_t smem, cudaStream_t st) {
  switch (CL) {
    case 1: return launch_topk2_cfg<NT, 1, BITS1>(a, rows, smem, st);
    case 2: return launch_topk2_cfg<NT, 2, BITS1>(a, rows, smem, st);
    case 4: return launch_topk2_cfg<NT, 4, BITS1>(a, rows, smem, st);
    case 8: return launch_topk2_cfg<NT, 8, BITS1>(a, rows, smem, st);
    default: return launch_topk2_cfg<NT, 16, BITS1>(a, rows, smem, st);
  }
}

// One CTA per row up to 32768 entries, longer rows over a cluster of 8 or 16
// CTAs (rows up to 16 x 32768 entries); 1024 threads per CTA when few CTAs
// run, else 512.  `hist` (optional): per-row histograms of the first
// IDX_HBITS key bits of the visible scores, built by the index kernel.
csa_status_t launch_topk2(const float* scores, int32_t* idx, int rows, int Tq, int N, int k, int m,
                          int q_pos0, uint32_t* hist, cudaStream_t st) {
  int CL = 1;
  if (N > 32768) {
    CL = 8;
    while (CL < 16 && (long long)CL * 32768 < N) CL <<= 1;
  } else if (hist && N > 8192 && (long long)rows * 8 <= 2LL * sm_count()) {
    CL = 8;   // few decode rows: spread the sweeps over 8 CTAs (measured faster than 1 or 16)
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
  csa::Topk2Args a{scores, idx, Tq, N, k, m, q_pos0, slice, cand_cap, hist};
  const bool wide = (long long)rows * CL <= 2LL * sm_count();
  if (hist) return wide ? launch_topk2_nt<1024, csa::IDX_HBITS>(a, CL, rows, smem, st)
                        : launch_topk2_nt<512, csa::IDX_HBITS>(a, CL, rows, smem, st);
  return wide ? launch_topk2_nt<1024, csa::TK2_BITS1>(a, CL, rows, smem, st)
              : launch_topk2_nt<512, csa::TK2_BITS1>(a, CL, rows, smem, st);
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
csa_status_t csa_compress(const void* Ca, const void* Cb, const void* Za, const void* Zb,
                          const float* Ba, const float* Bb, void* out, int B, int T, int d,
                          int m, int dtype, void* stream) {
  const int overlap = (Cb != nullptr) ? 1 : 0;
  if ((Cb == nullptr) != (Zb == nullptr)) return CSA_ERR_INVALID_ARG;
  if (B < 0 || T < 0 || d <= 0 || m <= 0 || m > 4096) return CSA_ERR_INVALID_ARG;
  if (dtype != CSA_DT_F32 && dtype != CSA_DT_BF16) return CSA_ERR_UNSUPPORTED;
  const int vec = dtype == CSA_DT_BF16 ? 8 : 4;
  if (d % vec || d / vec > 256) return CSA_ERR_UNSUPPORTED;
  if (B == 0 || T / m == 0) return CSA_OK;   // nothing to compress (outputs may be empty)
  if (!Ca || !Za || !out) return CSA_ERR_INVALID_ARG;
  const void* ptrs[] = {Ca, Cb, Za, Zb, out};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return CSA_ERR_INVALID_ARG;
  if ((Ba && !aligned(Ba, 4)) || (Bb && !aligned(Bb, 4))) return CSA_ERR_INVALID_ARG;
  const int N = T / m;
  if (B == 0 || N == 0) return CSA_OK;
  csa::CompressArgs a;
  a.Ca = Ca; a.Cb = Cb; a.Za = Za; a.Zb = Zb; a.Ba = Ba; a.Bb = Bb; a.out = out;
  a.B = B; a.T = T; a.d = d; a.m = m; a.N = N; a.overlap = overlap;
  a.vecs = d / vec;
  int rows = overlap ? 2 * m : m;
  int groups = 256 / a.vecs;
  if (groups > rows) groups = rows;
  if (groups < 1) groups = 1;
  a.groups = groups;
  dim3 grid(N, B);
  dim3 block(a.vecs * groups);
  size_t smem = (size_t)groups * a.vecs * 3 * vec * sizeof(float);
  {
    cudaError_t e = dtype == CSA_DT_BF16
                        ? launch_ex(csa::compress_kernel<__nv_bfloat16>, grid, block, smem, S(stream), 1, a)
                        : launch_ex(csa::compress_kernel<float>, grid, block, smem, S(stream), 1, a);
    if (e != cudaSuccess) return cuda_fail(e, "csa_compress launch");
  }
  return CSA_OK;
}

// ---------------------------------------------------------------------------
static csa_status_t index_impl(const void* qI, const void* qI_sf, const float* w, const void* K,
                              const void* K_sf, float* scores, int B, int Tq, int N, int H, int c,
                              int m, int q_pos0, int dtype, uint32_t* hist, void* stream) {
  if (B < 0 || Tq < 0 || N < 0 || H <= 0 || c <= 0 || m <= 0 || q_pos0 < 0)
    return CSA_ERR_INVALID_ARG;
  if (B == 0 || Tq == 0 || N == 0) return CSA_OK;
  if (!qI || !w || !K || !scores) return CSA_ERR_INVALID_ARG;
  if (dtype == CSA_DT_F32) {
    if (c > 256) return CSA_ERR_UNSUPPORTED;
    csa::IndexF32Args a{reinterpret_cast<const float*>(qI), w, reinterpret_cast<const float*>(K),
                        scores, Tq, N, H, c, m, q_pos0};
    dim3 grid((N + 7) / 8, B * Tq);
    cudaError_t e = launch_ex(csa::index_f32_kernel, grid, dim3(256), 0, S(stream), 1, a);
    if (e != cudaSuccess) return cuda_fail(e, "csa_index f32 launch");
    return CSA_OK;
  }
  if (dtype == CSA_DT_BF16) {
    if (!aligned(qI, 16) || !aligned(K, 16) || !aligned(w, 4) || !aligned(scores, 4))
      return CSA_ERR_INVALID_ARG;
    if (H == 64 && c == 128)
      return launch_index_tc<64, 128>(qI, w, K, scores, B, Tq, N, m, q_pos0, hist, S(stream));
    if (H == 64 && c == 64)
      return launch_index_tc<64, 64>(qI, w, K, scores, B, Tq, N, m, q_pos0, hist, S(stream));
    if (H == 32 && c == 128)
      return launch_index_tc<32, 128>(qI, w, K, scores, B, Tq, N, m, q_pos0, hist, S(stream));
    if (H == 128 && c == 128)
      return launch_index_tc<128, 128>(qI, w, K, scores, B, Tq, N, m, q_pos0, hist, S(stream));
    return CSA_ERR_UNSUPPORTED;
  }
  if (dtype == CSA_DT_E2M1_BLOCK16) {
    if (!qI_sf || !K_sf) return CSA_ERR_INVALID_ARG;
    if (!aligned(qI, 16) || !aligned(K, 16) || !aligned(qI_sf, 16) || !aligned(K_sf, 16) ||
        !aligned(w, 4) || !aligned(scores, 4))
      return CSA_ERR_INVALID_ARG;
    if (c != csa::FP4_C) return CSA_ERR_UNSUPPORTED;
    if (H == 64)
      return launch_index_fp4<64>(qI, qI_sf, w, K, K_sf, scores, B, Tq, N, m, q_pos0, hist, S(stream));
    if (H == 32)
      return launch_index_fp4<32>(qI, qI_sf, w, K, K_sf, scores, B, Tq, N, m, q_pos0, hist, S(stream));
    if (H == 128)
      return launch_index_fp4<128>(qI, qI_sf, w, K, K_sf, scores, B, Tq, N, m, q_pos0, hist, S(stream));
    return CSA_ERR_UNSUPPORTED;
  }
  return CSA_ERR_UNSUPPORTED;
}

csa_status_t csa_index(const void* qI, const void* qI_sf, const float* w, const void* K,
                       const void* K_sf, float* scores, int B, int Tq, int N, int H, int c,
                       int m, int q_pos0, int dtype, void* stream) {
  return index_impl(qI, qI_sf, w, K, K_sf, scores, B, Tq, N, H, c, m, q_pos0, dtype, nullptr, stream);
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
                            const void* K_sf, float* scores, int32_t* idx, int B, int Tq, int N,
                            int H, int c, int m, int q_pos0, int k, int dtype, void* ws,
                            size_t ws_bytes, void* stream) {
  if (k < 1 || k > 4096) return CSA_ERR_INVALID_ARG;
  if (!index_topk_fused(B, Tq, N, dtype)) {
    csa_status_t st = csa_index(qI, qI_sf, w, K, K_sf, scores, B, Tq, N, H, c, m, q_pos0, dtype, stream);
    if (st != CSA_OK) return st;
    return csa_topk(scores, idx, B, Tq, N, k, m, q_pos0, stream);
  }
  if (!idx || !aligned(idx, 4)) return CSA_ERR_INVALID_ARG;
  const size_t need = csa_index_topk_workspace_size(B, Tq, N, dtype);
  if (!ws || ws_bytes < need || !aligned(ws, 16)) return CSA_ERR_WORKSPACE;
  // the histograms start zero (caller's first use) and the selector clears each
  // row's after reading it, so no clearing pass runs here
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws);
  csa_status_t st = index_impl(qI, qI_sf, w, K, K_sf, scores, B, Tq, N, H, c, m, q_pos0, dtype, hist, stream);
  if (st != CSA_OK) return st;
  return launch_topk2(scores, idx, B * Tq, Tq, N, k, m, q_pos0, hist, S(stream));
}

// ---------------------------------------------------------------------------
csa_status_t csa_topk(const float* scores, int32_t* idx, int B, int Tq, int N, int k, int m,
                      int q_pos0, void* stream) {
  if (B < 0 || Tq < 0 || N < 0 || k < 1 || k > 4096 || m <= 0 || q_pos0 < 0)
    return CSA_ERR_INVALID_ARG;
  if (B == 0 || Tq == 0) return CSA_OK;
  if (!idx || (N > 0 && !scores)) return CSA_ERR_INVALID_ARG;
  if (!aligned(scores, 4) || !aligned(idx, 4)) return CSA_ERR_INVALID_ARG;
  const int rows = B * Tq;
  // few long decode rows up to 32768 entries: 8-bit radix passes over a 16-CTA
  // cluster; everything else up to 16 x 32768 entries: the candidate-filtering
  // selector (measured faster there: many short rows, and rows past 32768)
  if (!(N > 8192 && N <= 32768 && rows < 64) && N <= 16 * 32768)
    return launch_topk2(scores, idx, rows, Tq, N, k, m, q_pos0, nullptr, S(stream));
  // rows longer than 16 slices of 32768 keys: 8-bit radix passes over up to 16 SMs
  int CL = 1;
  if (N > 8192 && rows < 64) CL = rows <= 9 ? 16 : 8;
  int slice = (N + CL - 1) / CL;
  slice = (slice + 3) & ~3;
  const size_t smem = (size_t)slice * sizeof(uint32_t);
  if (smem > 200 * 1024) return CSA_ERR_UNSUPPORTED;
  csa::TopkArgs a{scores, idx, Tq, N, k, m, q_pos0, slice};
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

// ---------------------------------------------------------------------------
static csa_status_t attend_common(const void* q, csa_kv_t ent, const int32_t* idx, csa_kv_t win,
                                  const float* sink, void* out, int B, int Tq, int N, int k,
                                  int T_win, int win_base, int n_h, int d, int r, int m, int n_win,
                                  int q_pos0, float rope_base, void* ws, size_t ws_bytes,
                                  void* stream, int dense) {
  if (B < 0 || Tq < 0 || N < 0 || T_win < 0 || n_h <= 0 || d <= 0 || r < 0 || r > d || (r & 1) ||
      r > 128 || m <= 0 || n_win <= 0 || q_pos0 < 0 || win_base < 0 || !(rope_base > 0.f))
    return CSA_ERR_INVALID_ARG;
  if (!dense && (k < 1 || k > 4096)) return CSA_ERR_INVALID_ARG;
  if (N > 0 && !ent.data) return CSA_ERR_INVALID_ARG;
  if (B == 0 || Tq == 0) return CSA_OK;
  if (!q || !sink || !out || !win.data) return CSA_ERR_INVALID_ARG;
  if (!dense && !idx) return CSA_ERR_INVALID_ARG;
  // every window position of every query row must lie in the window buffer
  const long long t_first = q_pos0, t_last = (long long)q_pos0 + Tq - 1;
  const long long w_lo = t_first - n_win + 1 < 0 ? 0 : t_first - n_win + 1;
  if (w_lo < win_base || t_last >= (long long)win_base + T_win) return CSA_ERR_INVALID_ARG;
  (void)ws; (void)ws_bytes;
  const RopeFreqs rf = make_rope(r, rope_base);
  // q dtype is implied by the kv dtype for the tensor-core path; float32 here
  if (ent.dtype == CSA_DT_F32 && win.dtype == CSA_DT_F32) {
    if (d > 512 || (size_t)n_h * d > 16384) return CSA_ERR_UNSUPPORTED;
    csa::AttendF32Args a;
    a.q = reinterpret_cast<const float*>(q);
    a.ent = reinterpret_cast<const float*>(ent.data);
    a.idx = dense ? nullptr : idx;
    a.win = reinterpret_cast<const float*>(win.data);
    a.sink = sink;
    a.out = reinterpret_cast<float*>(out);
    a.Tq = Tq; a.N = N; a.k = dense ? 0 : k; a.T_win = T_win; a.win_base = win_base;
    a.n_h = n_h; a.d = d; a.r = r; a.m = m; a.n_win = n_win; a.q_pos0 = q_pos0;
    a.dense = dense;
    a.inv_sqrt_d = (float)(1.0 / std::sqrt((double)d));
    a.rf = rf;
    const size_t smem = ((size_t)2 * n_h * d + d + 5 * n_h) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(csa::attend_f32_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "csa_attend f32 attr");
    e = launch_ex(csa::attend_f32_kernel, dim3(B * Tq), dim3(csa::ATT_F32_THREADS), smem, S(stream), 1, a);
    if (e != cudaSuccess) return cuda_fail(e, "csa_attend f32 launch");
    return CSA_OK;
  }
  if (!tc_attend_shape(n_h, d, r, ent.dtype) || ent.dtype != win.dtype) return CSA_ERR_UNSUPPORTED;
  const int mixed = ent.dtype == CSA_DT_E4M3_BF16ROPE;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(win.data, 16) || (N > 0 && !aligned(ent.data, 16)))
    return CSA_ERR_INVALID_ARG;
  if (mixed && (!win.scale || !win.rope || !aligned(win.rope, 16) ||
                (N > 0 && (!ent.scale || !ent.rope || !aligned(ent.rope, 16)))))
    return CSA_ERR_INVALID_ARG;
  const AttPlan p = plan_attend(B, Tq, N, k, T_win, n_h, m, n_win, q_pos0, dense, mixed);
  if (p.bytes > 0 && (!ws || ws_bytes < p.bytes || !aligned(ws, 256))) return CSA_ERR_WORKSPACE;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  csa::AttendTcArgs a;
  memset(&a, 0, sizeof(a));
  a.q = reinterpret_cast<const __nv_bfloat16*>(q);
  a.ent = ent.data; a.ent_scale = ent.scale;
  a.ent_rope = reinterpret_cast<const __nv_bfloat16*>(ent.rope);
  a.win = win.data; a.win_scale = win.scale;
  a.win_rope = reinterpret_cast<const __nv_bfloat16*>(win.rope);
  a.idx = dense ? nullptr : idx;
  a.sink = sink;
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.B = B; a.Tq = Tq; a.N = N; a.k = dense ? 0 : k; a.T_win = T_win; a.win_base = win_base;
  a.n_h = n_h; a.m = m; a.n_win = n_win; a.q_pos0 = q_pos0;
  a.HG = p.HG; a.nch = p.nch; a.chunk_rows = p.chunk_rows; a.items = p.items;
  a.rotate_rows = p.rotate_rows; a.kv_mixed = mixed;
  a.cl_reduce = p.cl_reduce;
  a.rel_rope = p.rel_rope;
  if ((long long)B * N >= 0x7fffffffLL || (long long)B * T_win >= 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
  a.rf = rf;
  cudaStream_t st = S(stream);
  if (!p.rotate_rows) {
    // rotate the RoPE dims of every stored row once
    csa::RotateArgs ra;
    ra.rf = rf;
    if (N > 0) {
      ra.src = reinterpret_cast<const __nv_bfloat16*>(ent.data);
      ra.dst = reinterpret_cast<__nv_bfloat16*>(wsb + p.off_rot_ent);
      ra.rows = (long long)B * N; ra.rows_per_b = N; ra.m = m; ra.base = 0;
      cudaError_t e = launch_ex(csa::rope_rotate_rows_kernel, dim3((unsigned)((ra.rows * 64 + 255) / 256)),
                                dim3(256), 0, st, 1, ra);
      if (e != cudaSuccess) return cuda_fail(e, "csa_attend rotate entries");
      a.ent = ra.dst;
    }
    ra.src = reinterpret_cast<const __nv_bfloat16*>(win.data);
    ra.dst = reinterpret_cast<__nv_bfloat16*>(wsb + p.off_rot_win);
    ra.rows = (long long)B * T_win; ra.rows_per_b = T_win; ra.m = 0; ra.base = win_base;
    {
      cudaError_t e = launch_ex(csa::rope_rotate_rows_kernel, dim3((unsigned)((ra.rows * 64 + 255) / 256)),
                                dim3(256), 0, st, 1, ra);
      if (e != cudaSuccess) return cuda_fail(e, "csa_attend rotate window");
    }
    a.win = ra.dst;
  }
  if (p.nch > 1 && !p.cl_reduce) {
    a.part_o = reinterpret_cast<float*>(wsb + p.off_part_o);
    a.part_ml = reinterpret_cast<float*>(wsb + p.off_part_ml);
  }
  CUtensorMap tmq;
  memset(&tmq, 0, sizeof(tmq));
  if (!tmap_bf16_3d(&tmq, q, csa::ATT_D, (uint64_t)B * Tq * n_h, 1, (uint64_t)csa::ATT_D * 2,
                    (uint64_t)B * Tq * n_h * csa::ATT_D * 2, 64, csa::ATT_HG))
    return CSA_ERR_UNSUPPORTED;
  const int smem = csa::AttSmem::BYTES;
  cudaError_t e = cudaFuncSetAttribute(csa::attend_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "csa_attend tc attr");
  const int sms = sm_count();
  const int grid = p.items < sms ? p.items : sms;
  if (p.cl_reduce && p.nch > 8) {
    e = cudaFuncSetAttribute(csa::attend_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_fail(e, "csa_attend cluster attr");
  }
  e = launch_ex(csa::attend_tc_kernel, dim3(grid), dim3(csa::ATT_THREADS), smem, st,
                p.cl_reduce ? p.nch : 1, tmq, a);
  if (e != cudaSuccess) return cuda_fail(e, "csa_attend tc launch");
  if (p.nch > 1 && !p.cl_reduce) {
    csa::CombineArgs ca;
    ca.part_o = a.part_o; ca.part_ml = a.part_ml; ca.sink = sink; ca.out = a.out;
    ca.Tq = Tq; ca.n_h = n_h; ca.HG = p.HG; ca.nch = p.nch; ca.q_pos0 = q_pos0; ca.rf = rf;
    ca.rel_rope = p.rel_rope;
    const size_t cmb_smem = (size_t)p.nch * csa::ATT_HG * 2 * sizeof(float);
    if (cmb_smem > 48 * 1024) {
      e = cudaFuncSetAttribute(csa::attend_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)cmb_smem);
      if (e != cudaSuccess) return cuda_fail(e, "csa_attend combine attr");
    }
    e = launch_ex(csa::attend_combine_kernel,
                  dim3((unsigned)((size_t)B * Tq * p.HG * (csa::ATT_D / csa::CMB_DIMS))),
                  dim3(csa::CMB_THREADS), cmb_smem, st, 1, ca);
    if (e != cudaSuccess) return cuda_fail(e, "csa_attend combine launch");
  }
  return CSA_OK;
}

csa_status_t csa_attend(const void* q, csa_kv_t entries, const int32_t* idx, csa_kv_t win,
                        const float* sink, void* out, int B, int Tq, int N, int k, int T_win,
                        int win_base, int n_h, int d, int r, int m, int n_win, int q_pos0,
                        float rope_base, void* ws, size_t ws_bytes, void* stream) {
  return attend_common(q, entries, idx, win, sink, out, B, Tq, N, k, T_win, win_base, n_h, d, r,
                       m, n_win, q_pos0, rope_base, ws, ws_bytes, stream, 0);
}

csa_status_t hca_attend(const void* q, csa_kv_t entries, csa_kv_t win, const float* sink,
                        void* out, int B, int Tq, int N, int T_win, int win_base, int n_h, int d,
                        int r, int m, int n_win, int q_pos0, float rope_base, void* ws,
                        size_t ws_bytes, void* stream) {
  return attend_common(q, entries, nullptr, win, sink, out, B, Tq, N, 0, T_win, win_base, n_h, d,
                       r, m, n_win, q_pos0, rope_base, ws, ws_bytes, stream, 1);
}

size_t csa_attend_workspace_size(int B, int Tq, int N, int k, int T_win, int n_h, int d, int r,
                                 int m, int n_win, int q_pos0, int q_dtype, int kv_dtype,
                                 int is_hca) {
  (void)q_dtype;
  if (B <= 0 || Tq <= 0 || n_h <= 0 || m <= 0 || N < 0) return 0;
  if (!tc_attend_shape(n_h, d, r, kv_dtype)) return 0;
  return plan_attend(B, Tq, N, is_hca ? 0 : k, T_win, n_h, m, n_win, q_pos0, is_hca ? 1 : 0,
                     kv_dtype == CSA_DT_E4M3_BF16ROPE ? 1 : 0).bytes;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// csa_attend_noalloc: csa_attend for callers that cannot allocate device
// memory.  Its scratch is one fixed array in this library's device image.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_attend_noalloc_scratch[CSA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoallocMaxDevices] = {};

// Device address of the scratch array on the current device.  The array's
// name in host code is only a host-side handle, so the address is looked up
// once per device (with that device current) and cached.
csa_status_t noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "csa_attend_noalloc get device");
  if (dev < 0 || dev >= kNoallocMaxDevices) return CSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attend_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "csa_attend_noalloc scratch address");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return CSA_OK;
}

}  // namespace

extern "C" csa_status_t csa_attend_noalloc(const void* q, csa_kv_t entries, const int32_t* idx,
                                           csa_kv_t win, const float* sink, void* out, int B,
                                           int Tq, int N, int k, int T_win, int win_base, int n_h,
                                           int d, int r, int m, int n_win, int q_pos0,
                                           float rope_base, void* stream) {
  const size_t need = csa_attend_workspace_size(B, Tq, N, k, T_win, n_h, d, r, m, n_win, q_pos0,
                                                CSA_DT_BF16, entries.dtype, 0);
  if (need > CSA_NOALLOC_SCRATCH_BYTES) {
    snprintf(g_cuda_msg, sizeof(g_cuda_msg),
             "csa_attend_noalloc: these sizes need %zu scratch bytes, above the fixed %zu", need,
             (size_t)CSA_NOALLOC_SCRATCH_BYTES);
    return CSA_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  if (need > 0) {
    const csa_status_t s = noalloc_scratch(&ws);
    if (s != CSA_OK) return s;
  }
  return attend_common(q, entries, idx, win, sink, out, B, Tq, N, k, T_win, win_base, n_h, d, r,
                       m, n_win, q_pos0, rope_base, ws, need > 0 ? (size_t)CSA_NOALLOC_SCRATCH_BYTES : 0,
                       stream, 0);
}
