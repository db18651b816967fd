// Softmax-weighted block compression (CSA overlapped, HCA non-overlapped).
//
// DeepSeek-V4 report (Chinese translation, blog.uika.cn) §2.3.1 compression
// equations and §2.3.2: entry i, channel c is sum_j S[j,c] * C[j,c] with
// S = softmax over the entry's rows of (Z + bias).  CSA rows: a-rows of block
// i and b-rows of block i-1 (none for i = 0); HCA rows: the block's m rows.
//
// Optional epilogue per entry: RMSNorm (§2.3.3) and RoPE of the last r dims
// at the entry's position, so that the attention can take it pre-rotated.
//
// HBM streaming reduction: one CTA per compressed entry.  Thread (v, g) owns
// one 16-byte channel vector v and visits rows g, g+G, ... with an online
// softmax (running max, running sum, running weighted sum per channel); the G
// row groups merge through shared memory at the end.  Every input byte is read
// once with 16-byte coalesced loads.
#pragma once
#include "common.cuh"

namespace csa {

template <typename T>
struct VecTraits;
template <> struct VecTraits<__nv_bfloat16> {
  static constexpr int N = 8;
  static CSA_DEVINL void load(const __nv_bfloat16* p, float* f) {
    bf16x8_to_f(__ldg(reinterpret_cast<const uint4*>(p)), f);
  }
  static CSA_DEVINL void store(__nv_bfloat16* p, const float* f) {
    *reinterpret_cast<uint4*>(p) = f_to_bf16x8(f);
  }
};
template <> struct VecTraits<float> {
  static constexpr int N = 4;
  static CSA_DEVINL void load(const float* p, float* f) {
    float4 v = __ldg(reinterpret_cast<const float4*>(p));
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  static CSA_DEVINL void store(float* p, const float* f) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};

struct CompressArgs {
  const void* Ca; const void* Cb; const void* Za; const void* Zb;
  const float* Ba; const float* Bb;
  void* out;
  int B, T, d, m, N;
  int overlap;      // 1 = CSA (b-rows of the previous block join), 0 = HCA
  int vecs;         // d / VEC
  int groups;       // row groups G (blockDim.x = vecs * groups)
  // optional epilogue on each compressed entry (applied in this order):
  int rms_norm;               // 1 = x / sqrt(mean(x^2) + eps) [* norm_weight]
  const float* norm_weight;   // [d] or null
  float norm_eps;
  int rope_dims;              // r > 0: rotate the last r dims at the entry's position m(i+1)-1
  RopeFreqs rf;
  // paged output (no table: out is [B, N, d]): entry i >= out_first of batch
  // row b goes to logical row out_entry0[b] + i - out_first of the pool; a
  // negative out_entry0[b] writes nothing for that batch row
  RowPages out_pg;
  const int32_t* out_entry0;
  int out_first;
};

template <typename T>
__global__ void __launch_bounds__(256) compress_kernel(CompressArgs a) {
  pdl_enter();
  using V = VecTraits<T>;
  constexpr int VEC = V::N;
  const int i = blockIdx.x;            // entry
  const int b = blockIdx.y;            // batch row
  const int v = threadIdx.x % a.vecs;  // channel vector
  const int g = threadIdx.x / a.vecs;  // row group
  const int c0 = v * VEC;

  // where this entry goes (the whole CTA leaves at once when it writes nothing)
  long long li = i;                    // logical entry index: RoPE position m(li+1)-1
  long long orow = (long long)b * a.N + i;
  if (a.out_pg.table) {
    const long long e0 = a.out_entry0 ? (long long)__ldg(a.out_entry0 + b) : 0LL;
    if (e0 < 0 || i < a.out_first) return;
    li = e0 + (i - a.out_first);
    orow = page_row(a.out_pg, b, li, 0);
    if (orow < 0) {
      if (threadIdx.x == 0) csa_flag_error(ERRBIT_BAD_INDEX);   // block outside the pool
      return;
    }
  }

  const size_t seq = (size_t)b * a.T * a.d;
  const T* Ca = reinterpret_cast<const T*>(a.Ca) + seq;
  const T* Za = reinterpret_cast<const T*>(a.Za) + seq;
  const T* Cb = a.overlap ? reinterpret_cast<const T*>(a.Cb) + seq : nullptr;
  const T* Zb = a.overlap ? reinterpret_cast<const T*>(a.Zb) + seq : nullptr;

  float mx[VEC], sum[VEC], acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) { mx[e] = -INFINITY; sum[e] = 0.f; acc[e] = 0.f; }

  // rows 0..m-1: a-rows of block i; rows m..2m-1: b-rows of block i-1
  const int nrows = (a.overlap && i > 0) ? 2 * a.m : a.m;
  for (int j = g; j < nrows; j += a.groups) {
    const bool is_a = j < a.m;
    const int jj = is_a ? j : j - a.m;
    const size_t tok = is_a ? (size_t)a.m * i + jj : (size_t)a.m * (i - 1) + jj;
    float z[VEC], cv[VEC];
    V::load((is_a ? Za : Zb) + tok * a.d + c0, z);
    V::load((is_a ? Ca : Cb) + tok * a.d + c0, cv);
    const float* bias = is_a ? a.Ba : a.Bb;
    if (bias) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) z[e] += __ldg(bias + (size_t)jj * a.d + c0 + e);
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      float nm = fmaxf(mx[e], z[e]);
      float sc = __expf(mx[e] - nm);       // 0 on the first row (mx = -inf)
      float p = __expf(z[e] - nm);
      sum[e] = sum[e] * sc + p;
      acc[e] = acc[e] * sc + p * cv[e];
      mx[e] = nm;
    }
  }

  // merge the row groups: group 0 of each vector gathers the others
  extern __shared__ float sm[];                  // [groups][vecs][3*VEC], then [vecs]
  float* mine = sm + ((size_t)g * a.vecs + v) * 3 * VEC;
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    mine[e] = mx[e]; mine[VEC + e] = sum[e]; mine[2 * VEC + e] = acc[e];
  }
  __syncthreads();
  const bool owner = g == 0;                     // threads 0 .. vecs-1 hold the entry's channels
  float res[VEC];
  if (owner) {
    for (int gg = 1; gg < a.groups; ++gg) {
      const float* o = sm + ((size_t)gg * a.vecs + v) * 3 * VEC;
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        float om = o[e];
        if (om == -INFINITY) continue;           // group saw no rows
        float nm = fmaxf(mx[e], om);
        float s0 = __expf(mx[e] - nm), s1 = __expf(om - nm);
        sum[e] = sum[e] * s0 + o[VEC + e] * s1;
        acc[e] = acc[e] * s0 + o[2 * VEC + e] * s1;
        mx[e] = nm;
      }
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) res[e] = acc[e] / sum[e];
  }
  if (a.rms_norm) {
    // RMSNorm of the entry (DeepSeek-V4 report, Chinese translation, §2.3.3:
    // the compressed entries are RMS-normalised before core attention).  Each
    // owner's sum of squares goes to shared memory and every owner adds them
    // in the same order, so the result does not depend on scheduling.
    float* red = sm + (size_t)a.groups * a.vecs * 3 * VEC;   // [vecs]
    if (owner) {
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < VEC; ++e) ss = fmaf(res[e], res[e], ss);
      red[v] = ss;
    }
    __syncthreads();
    if (owner) {
      float tot = 0.f;
      for (int w = 0; w < a.vecs; ++w) tot += red[w];
      const float sc = rsqrtf(tot / (float)a.d + a.norm_eps);
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        res[e] *= sc * (a.norm_weight ? __ldg(a.norm_weight + c0 + e) : 1.f);
    }
  }
  if (!owner) return;
  if (a.rope_dims > 0 && c0 >= a.d - a.rope_dims) {
    // RoPE of the last r dims at the entry's position (the last token it
    // summarises), so consumers can take the entry as already rotated
    const long long pos = (long long)a.m * (li + 1) - 1;
    const int j0 = (c0 - (a.d - a.rope_dims)) >> 1;
#pragma unroll
    for (int p = 0; p < VEC / 2; ++p) {
      float cs, sn;
      rope_cos_sin(pos, a.rf.F[j0 + p], cs, sn);
      const float x0 = res[2 * p], x1 = res[2 * p + 1];
      res[2 * p] = x0 * cs - x1 * sn;
      res[2 * p + 1] = x0 * sn + x1 * cs;
    }
  }
  T* out = reinterpret_cast<T*>(a.out) + (size_t)orow * a.d + c0;
  V::store(out, res);
}

}  // namespace csa
