// float32 CUDA-core kernels for the lightning indexer and the core attention.
//
// These serve float32 workloads (and shapes too small for tensor-core tiles,
// e.g. 4 query heads of dim 128).  They follow the same definitions as the
// tensor-core kernels: DeepSeek-V4 report (Chinese translation,
// blog.uika.cn) §2.3.1 indexer score and shared-KV MQA, §2.3.3 partial RoPE
// with inverse rotation of the output, sliding window and attention sink.
#pragma once
#include "common.cuh"

namespace csa {

// ----------------------------------------------------------------------------
// indexer: one warp per (row, entry s); lanes split the H*c products
// ----------------------------------------------------------------------------
struct IndexF32Args {
  const float* q; const float* w; const float* K; void* scores;
  const int32_t* q_pos;            // [B, Tq] (null: t = i)
  int scores_bf16;                 // 1 = scores stored as bf16
  RowPages k_pg;                   // paged keys (no table: flat)
  int Tq, N, H, c, m;
};

__global__ void __launch_bounds__(256) index_f32_kernel(IndexF32Args a) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int row = blockIdx.y;                      // b * Tq + i
  if (gw >= a.N) return;
  const int s = (int)gw;
  const int b = row / a.Tq, i = row % a.Tq;
  const long long t = query_pos(a.q_pos, row, i);
  if (t < 0 && s == 0 && lane == 0) csa_flag_error(ERRBIT_BAD_INDEX);
  const size_t out = (size_t)row * a.N + s;
  if (t < 0 || (long long)(s + 1) * a.m > t + 1) {   // not visible
    if (lane == 0) {
      if (a.scores_bf16) reinterpret_cast<__nv_bfloat16*>(a.scores)[out] = __float2bfloat16_rn(-INFINITY);
      else reinterpret_cast<float*>(a.scores)[out] = -INFINITY;
    }
    return;
  }
  const float* qr = a.q + (size_t)row * a.H * a.c;
  const long long krow = page_row(a.k_pg, b, s, a.N);
  if (krow < 0) {                                    // block outside the pool
    if (lane == 0) csa_flag_error(ERRBIT_BAD_INDEX);
    return;
  }
  const float* kr = a.K + (size_t)krow * a.c;
  const float* wr = a.w + (size_t)row * a.H;
  float acc = 0.f;
  for (int h = 0; h < a.H; ++h) {
    float dot = 0.f;
    for (int j = lane; j < a.c; j += 32) dot = fmaf(qr[(size_t)h * a.c + j], kr[j], dot);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    acc = fmaf(wr[h], fmaxf(dot, 0.f), acc);
  }
  if (lane == 0) {
    if (a.scores_bf16) reinterpret_cast<__nv_bfloat16*>(a.scores)[out] = __float2bfloat16_rn(acc);
    else reinterpret_cast<float*>(a.scores)[out] = acc;
  }
}

// ----------------------------------------------------------------------------
// attention: one CTA per query row; online softmax over the row set
// (selected compressed entries, then the window), float32 throughout.
// ----------------------------------------------------------------------------
struct AttendF32Args {
  const float* q; const float* ent; const int32_t* idx; const float* win; const float* sink;
  float* out;
  const int32_t* q_pos;            // [B, Tq] (null: t = i)
  const int32_t* win_base;         // [B] (null: 0)
  int Tq, N, k, T_win, n_h, d, r, m, n_win;
  int dense;        // 1 = HCA: every visible entry, idx unused
  int ent_rotated;  // 1 = entries stored with their RoPE dims already rotated
  RowPages ent_pg, win_pg;   // paged / ring row maps (no table: flat)
  float inv_sqrt_d;
  RopeFreqs rf;
};

constexpr int ATT_F32_THREADS = 256;

__global__ void __launch_bounds__(ATT_F32_THREADS) attend_f32_kernel(AttendF32Args a) {
  pdl_enter();
  extern __shared__ float sm[];
  const int row = blockIdx.x;                    // b * Tq + i
  const int b = row / a.Tq, i = row % a.Tq;
  const long long t = query_pos(a.q_pos, row, i);
  const long long wbase = window_base(a.win_base, b);
  const int nh = a.n_h, d = a.d, r = a.r;
  float* qs = sm;                                // [n_h][d] rotated queries
  float* acc = qs + (size_t)nh * d;              // [n_h][d]
  float* er = acc + (size_t)nh * d;              // [d] current rotated row
  float* lg = er + d;                            // [n_h] logits of the current row
  float* mrun = lg + nh;                         // [n_h] running max
  float* lrun = mrun + nh;                       // [n_h] running denominator
  float* scl = lrun + nh;                        // [n_h] rescale of acc for this row
  float* pw = scl + nh;                          // [n_h] weight of this row
  const int tid = threadIdx.x;
  const int lane = tid & 31, wid = tid >> 5, nw = ATT_F32_THREADS / 32;

  const float* qg = a.q + (size_t)row * nh * d;
  for (int x = tid; x < nh * d; x += ATT_F32_THREADS) {
    qs[x] = qg[x];
    acc[x] = 0.f;
  }
  for (int h = tid; h < nh; h += ATT_F32_THREADS) { mrun[h] = -INFINITY; lrun[h] = 0.f; }
  __syncthreads();
  // rotate the query's RoPE dims at position t
  for (int x = tid; x < nh * (r / 2); x += ATT_F32_THREADS) {
    const int h = x / (r / 2), j = x % (r / 2);
    float c, s;
    rope_cos_sin(t, a.rf.F[j], c, s);
    float* p = qs + (size_t)h * d + (d - r) + 2 * j;
    float x0 = p[0], x1 = p[1];
    p[0] = x0 * c - x1 * s;
    p[1] = x0 * s + x1 * c;
  }
  __syncthreads();

  // row list: [0, nsel) compressed entries, then the window tokens
  int nsel;
  const int32_t* irow = a.idx ? a.idx + (size_t)row * a.k : nullptr;
  int vis = t < 0 ? 0 : (int)min((long long)a.N, (t + 1) / a.m);
  if (t < 0 && tid == 0) csa_flag_error(ERRBIT_BAD_INDEX);
  nsel = t < 0 ? 0 : (a.dense ? vis : a.k);
  const long long w0 = max(0LL, t - a.n_win + 1);
  const int nwin = t < 0 ? 0 : (int)(t - w0 + 1);
  for (int jr = 0; jr < nsel + nwin; ++jr) {
    const float* src;
    long long pos;
    if (jr < nsel) {
      int s = a.dense ? jr : irow[jr];
      if (s < 0) continue;                       // uniform across the block
      if (s >= a.N) { if (tid == 0) csa_flag_error(ERRBIT_BAD_INDEX); continue; }
      const long long prow = page_row(a.ent_pg, b, s, a.N);
      if (prow < 0) { if (tid == 0) csa_flag_error(ERRBIT_BAD_INDEX); continue; }
      src = a.ent + (size_t)prow * d;
      pos = a.ent_rotated ? 0 : (long long)a.m * (s + 1) - 1;   // a turn by 0 leaves the row as stored
    } else {
      const long long tok = w0 + (jr - nsel);
      if (tok < wbase || tok >= wbase + a.T_win) {    // outside this batch row's window buffer
        if (tid == 0) csa_flag_error(ERRBIT_BAD_INDEX);
        continue;
      }
      const long long prow = page_row(a.win_pg, b, window_row(a.win_pg, tok, wbase, a.T_win), a.T_win);
      if (prow < 0) { if (tid == 0) csa_flag_error(ERRBIT_BAD_INDEX); continue; }
      src = a.win + (size_t)prow * d;
      pos = tok;
    }
    for (int x = tid; x < d; x += ATT_F32_THREADS) er[x] = src[x];
    __syncthreads();
    for (int j = tid; j < r / 2; j += ATT_F32_THREADS) {
      float c, s;
      rope_cos_sin(pos, a.rf.F[j], c, s);
      float* p = er + (d - r) + 2 * j;
      float x0 = p[0], x1 = p[1];
      p[0] = x0 * c - x1 * s;
      p[1] = x0 * s + x1 * c;
    }
    __syncthreads();
    for (int h = wid; h < nh; h += nw) {
      float dot = 0.f;
      for (int x = lane; x < d; x += 32) dot = fmaf(qs[(size_t)h * d + x], er[x], dot);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      if (lane == 0) {
        const float l = dot * a.inv_sqrt_d;
        const float nm = fmaxf(mrun[h], l);
        const float sc = expf(mrun[h] - nm);
        const float p = expf(l - nm);
        lrun[h] = lrun[h] * sc + p;
        mrun[h] = nm;
        scl[h] = sc;
        pw[h] = p;
      }
    }
    __syncthreads();
    for (int x = tid; x < nh * d; x += ATT_F32_THREADS) {
      const int h = x / d;
      acc[x] = acc[x] * scl[h] + pw[h] * er[x % d];
    }
    __syncthreads();
  }
  // sink joins the denominator, then normalise and rotate back by -t
  for (int x = tid; x < nh * d; x += ATT_F32_THREADS) {
    const int h = x / d;
    const float z = a.sink[h];
    const float M = fmaxf(mrun[h], z);
    const float den = lrun[h] * expf(mrun[h] - M) + expf(z - M);
    acc[x] = acc[x] * expf(mrun[h] - M) / den;
  }
  __syncthreads();
  for (int x = tid; x < nh * (r / 2); x += ATT_F32_THREADS) {
    const int h = x / (r / 2), j = x % (r / 2);
    float c, s;
    rope_cos_sin(-t, a.rf.F[j], c, s);
    float* p = acc + (size_t)h * d + (d - r) + 2 * j;
    float x0 = p[0], x1 = p[1];
    p[0] = x0 * c - x1 * s;
    p[1] = x0 * s + x1 * c;
  }
  __syncthreads();
  float* og = a.out + (size_t)row * nh * d;
  for (int x = tid; x < nh * d; x += ATT_F32_THREADS) og[x] = acc[x];
}

}  // namespace csa
