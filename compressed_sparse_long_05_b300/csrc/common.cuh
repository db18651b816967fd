// Shared device helpers for the CSA / HCA kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#define CSA_DEVINL __device__ __forceinline__

// Sticky device error word (one per device, in this library's module).
// Bit values: see the ERRBIT_* constants.
__device__ unsigned int g_csa_error_word;

enum : unsigned int {
  ERRBIT_TIMEOUT = 1u,      // a bounded mbarrier wait gave up
  ERRBIT_BAD_INDEX = 2u,    // an index >= N, a negative position, or a row outside its buffer or pool
  ERRBIT_TMEM = 4u,         // tensor-memory allocation returned an unusable address
  ERRBIT_HIST = 8u          // a key-digit histogram disagreed with the scores it describes
};

CSA_DEVINL void csa_flag_error(unsigned int bit) { atomicOr(&g_csa_error_word, bit); }

CSA_DEVINL long long csa_globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return (long long)t;
}

// ----------------------------------------------------------------------------
// Phase trace (built only into the traced library variant, -DCSA_TRACE): a
// kernel marks the SM clock at its phase boundaries for CTAs below
// CSA_TRACE_CTAS; the host reads the marks with csa_trace_read().  Marks
// record, they change no work.
// ----------------------------------------------------------------------------
#ifdef CSA_TRACE
namespace csa {
constexpr int CSA_TRACE_CTAS = 160;
constexpr int CSA_TRACE_SLOTS = 64;   // attention 0-31, index 32-47, top-k 48-63
__device__ long long g_csa_trace[CSA_TRACE_CTAS][CSA_TRACE_SLOTS];
__device__ int g_csa_trace_tile;   // which tile of a CTA the per-tile marks describe
}  // namespace csa
#define CSA_TRACE_TILE (csa::g_csa_trace_tile)
#define CSA_TRACE_MARK(slot)                                                         \
  do {                                                                               \
    if (blockIdx.x < csa::CSA_TRACE_CTAS) {                                               \
      long long c_;                                                                  \
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(c_));                           \
      csa::g_csa_trace[blockIdx.x][(slot)] = c_;                                          \
    }                                                                                \
  } while (0)
#define CSA_TRACE_WALL(slot)                                                         \
  do {                                                                               \
    if (blockIdx.x < csa::CSA_TRACE_CTAS) csa::g_csa_trace[blockIdx.x][(slot)] = csa_globaltimer(); \
  } while (0)
#else
#define CSA_TRACE_MARK(slot) do {} while (0)
#define CSA_TRACE_WALL(slot) do {} while (0)
#define CSA_TRACE_TILE 0
#endif

// Absolute token position of query row `row` = b * Tq + i: q_pos[row] when the
// caller passed positions, else i (causal prefill from token 0).
CSA_DEVINL long long query_pos(const int32_t* q_pos, long long row, int i) {
  return q_pos ? (long long)__ldg(q_pos + row) : (long long)i;
}
// Hint: bring the line of p into L1 (no wait; the first item's small reads
// issued at kernel entry so their latency overlaps the set-up).
CSA_DEVINL void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}
// Window buffer base token of batch row b (0 without a base array).
CSA_DEVINL long long window_base(const int32_t* win_base, int b) {
  return win_base ? (long long)__ldg(win_base + b) : 0LL;
}

// Paged rows (the block-table layout of the KV cache, DeepSeek-V4 report,
// Chinese translation, blog.uika.cn, §3.6.1): logical row j of sequence b sits
// in block table[b * max_blocks + j / block_rows] of a pool shared by every
// sequence, at row j % block_rows of that block.  No table: the flat layout,
// row b * rows + j.  ring (window buffers): token p is logical row p mod rows.
struct RowPages {
  const int32_t* table;
  int max_blocks, block_rows, num_blocks, ring;
  int shift;          // log2(block_rows) when it is a power of two, else -1
};

// Physical row of logical row j (0 <= j < 2^31) of sequence b, rows per
// sequence in the flat layout; -1 when the block-table entry is outside the
// pool (the caller flags it and leaves the row out).  32-bit arithmetic, and a
// shift for power-of-two blocks: one lane may map many rows.
CSA_DEVINL long long page_row(const RowPages& p, int b, long long j, long long rows) {
  if (!p.table) return (long long)b * rows + j;
  const unsigned int ju = (unsigned int)j;
  unsigned int blk_l, off;
  if (p.shift >= 0) {
    blk_l = ju >> p.shift;
    off = ju & ((1u << p.shift) - 1u);
  } else {
    blk_l = ju / (unsigned int)p.block_rows;
    off = ju - blk_l * (unsigned int)p.block_rows;
  }
  if (blk_l >= (unsigned int)p.max_blocks) return -1;
  const int blk = __ldg(p.table + (size_t)b * p.max_blocks + blk_l);
  if (blk < 0 || blk >= p.num_blocks) return -1;
  return (long long)blk * p.block_rows + off;
}

// Logical row of window token tok (tokens base .. base + rows - 1 present; tok
// and rows below 2^31).
CSA_DEVINL long long window_row(const RowPages& p, long long tok, long long base, long long rows) {
  return p.ring ? (long long)((unsigned int)tok % (unsigned int)rows) : tok - base;
}

// Programmatic dependent launch.  Every kernel lets the next launch in the
// stream start as early as possible (its prologue overlaps this grid's tail),
// and waits for the previous grid to complete and flush before its first global
// memory access.  Without a programmatic predecessor the wait returns at once.
CSA_DEVINL void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
CSA_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
CSA_DEVINL void pdl_enter() { pdl_launch_dependents(); pdl_wait(); }

// ----------------------------------------------------------------------------
// numeric helpers
// ----------------------------------------------------------------------------

template <typename T> struct Elem;
template <> struct Elem<float> {
  static CSA_DEVINL float to_f(float x) { return x; }
  static CSA_DEVINL float from_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static CSA_DEVINL float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static CSA_DEVINL __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// 8 bf16 <-> 8 float, through one 16-byte vector.
CSA_DEVINL void bf16x8_to_f(const uint4& v, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
CSA_DEVINL uint4 f_to_bf16x8(const float* f) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}
CSA_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ----------------------------------------------------------------------------
// RoPE angle from a fixed-point phase.
// The host stores, per frequency j, F_j = round(theta_j / (2*pi) * 2^64) as a
// uint64.  For an integer position p the rotation phase in revolutions is
// p * F_j / 2^64 modulo 1, which unsigned 64-bit multiplication gives exactly
// (wrap-around is the modulo).  Only its top 32 bits are needed: for
// F = F_hi 2^32 + F_lo they are |p| F_hi + hi32(|p| F_lo) modulo 2^32, three
// 32-bit operations.  Read as a signed fraction in [-1/2, 1/2) they give an
// angle in [-pi, pi) that the fast hardware sine/cosine evaluate to about 1e-6
// absolute, so the angle stays accurate at any position |p| < 2^31 (plain fp32
// p * theta would be off by up to 0.06 rad at 2^20).  A negative position
// turns the other way: the same cosine, the sine negated.
// ----------------------------------------------------------------------------
struct RopeFreqs {
  unsigned long long F[64];  // one per rotated pair; r/2 <= 64
  int half;                  // r / 2
};

CSA_DEVINL void rope_cos_sin(long long pos, unsigned long long F, float& c, float& s) {
  const unsigned int ap = (unsigned int)(pos < 0 ? -pos : pos);
  const unsigned int w = ap * (unsigned int)(F >> 32) + __umulhi(ap, (unsigned int)F);
  const float rev = (float)(int)w * 2.3283064365386963e-10f;   // * 2^-32
  __sincosf(6.283185307179586f * rev, &s, &c);
  if (pos < 0) s = -s;
}

// ----------------------------------------------------------------------------
// ordered keys for float radix selection: unsigned order == float order
// ----------------------------------------------------------------------------
CSA_DEVINL uint32_t float_to_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
