// Quantizer kernels: per-tensor amax (plain and after the 16-point random
// Hadamard transform), the DelayedScaling history/scale update, and the FP8,
// MXFP8 and NVFP4 quantizers that write the row-wise and column-wise
// (transposed) copies of a tensor from a single read.
//
// Every quantizer thread owns a register patch (16 or 32 consecutive rows of one
// 16- or 8-byte row vector), so the input is read from HBM exactly once for both
// copies, with all of a thread's loads in flight together and no shared-memory
// staging or block barriers.  All code-deciding arithmetic is IEEE fp32
// round-to-nearest-even (compiled with -fmad=false) so the codes are bit-identical
// to the definitions in te_gb300.h.
#include <cuda_bf16.h>
#include <string.h>

#include <mutex>

#include <type_traits>

#include "common.cuh"

namespace te {
namespace {

constexpr int kThreads = 256;

// ---- format conversions (hardware cvt, round-to-nearest-even, satfinite) --------------

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t cvt_e5m2x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}
// Two E2M1 codes: `lo` in bits 0-3, `hi` in bits 4-7.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t d;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// Value of a UE4M3 code (exact).
__device__ __forceinline__ float ue4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  if (e == 0) return static_cast<float>(m) * 0.001953125f;  // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// 16 fp32 values -> 16 FP8 codes in a uint4 (element i in byte i).
template <bool E5M2>
__device__ __forceinline__ uint4 pack_fp8_16(const float (&v)[16], float s) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float a = __fmul_rn(v[4 * j], s), b = __fmul_rn(v[4 * j + 1], s);
    const float c = __fmul_rn(v[4 * j + 2], s), d = __fmul_rn(v[4 * j + 3], s);
    const uint32_t p0 = E5M2 ? cvt_e5m2x2(a, b) : cvt_e4m3x2(a, b);
    const uint32_t p1 = E5M2 ? cvt_e5m2x2(c, d) : cvt_e4m3x2(c, d);
    w[j] = p0 | (p1 << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---- Philox4x32-10 (Salmon et al., SC'11) and stochastic E2M1 rounding ---------------

// Philox4x32-10 with its ten round keys given (k0[i] = seed_lo + i * 0x9E3779B9,
// k1[i] = seed_hi + i * 0xBB67AE85, the key schedule of the published definition): the
// kernels read them from their parameters, so no key bumps execute per call.
__device__ __forceinline__ uint4 philox4x32_10_rk(uint4 c, const uint32_t (&k0)[10], const uint32_t (&k1)[10]) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c.x;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c.z;
    c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ k0[i], static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ c.w ^ k1[i], static_cast<uint32_t>(p0));
  }
  return c;
}


// Four E2M1 codes with stochastic rounding (element i in bits 4i..4i+3).  The
// hardware conversion adds 16 random bits below the kept bit and truncates; the
// 32-bit word w feeds all four: P = (w[23:16] << 8) | w[7:0] drives elements 0
// (as is) and 1 (bit-reversed), Q = (w[31:24] << 8) | w[15:8] elements 2 and 3.
__device__ __forceinline__ uint32_t cvt_e2m1x4_rs(float e0, float e1, float e2, float e3, uint32_t w) {
  uint16_t d;
  asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;" : "=h"(d) : "f"(e3), "f"(e2), "f"(e1), "f"(e0), "r"(w));
  return d;
}

// ---- 16-point random Hadamard transform ----------------------------------------------------

__device__ __forceinline__ void rht16(float (&v)[16], uint32_t signs) {
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if ((signs >> j) & 1u) v[j] = -v[j];
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      const float a = v[i], b = v[i + h];
      v[i] = __fadd_rn(a, b);
      v[i + h] = __fsub_rn(a, b);
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], 0.25f);
}

// ---- packed fp32 pairs (two IEEE round-to-nearest operations per instruction) ----------------

__device__ __forceinline__ float2 f2neg(float2 a) { return make_float2(-a.x, -a.y); }
// Butterflies h = 1, 2, 4, 8 of the 16-point Hadamard transform on two columns at
// once (y[r] holds row r of both); the same operations in the same order as rht16
// (a - b is computed as a + (-b), which is the same rounded result).
template <int kLastH = 8>
__device__ __forceinline__ void hadamard16x2(float2 (&y)[16]) {
#pragma unroll
  for (int h = 1; h <= kLastH; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      const float2 a = y[i], b = y[i + h];
      y[i] = __fadd2_rn(a, b);
      y[i + h] = __fadd2_rn(a, f2neg(b));
    }
  }
}
// Sign-flip mask of row j for a word of two bf16 values (both flipped when bit j of signs is set).
__device__ __forceinline__ uint32_t rht_sign2(uint32_t signs, int j) { return (0u - ((signs >> j) & 1u)) & 0x80008000u; }

// ---- reductions -----------------------------------------------------------------------------

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
// Max over aligned groups of L consecutive lanes (L a power of two <= 32).
template <int L>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = 1; o < L; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
// Block-wide max, then one atomicMax on the (non-negative) fp32 bit pattern.
__device__ __forceinline__ void block_max_to(float v, float* out) {
  __shared__ float red[32];
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    v = (l < static_cast<int>(blockDim.x >> 5)) ? red[l] : 0.0f;
    v = warp_max(v);
    if (l == 0) atomicMax(reinterpret_cast<unsigned int*>(out), __float_as_uint(v));
  }
  __syncthreads();
}

// ---- register patches ---------------------------------------------------------------------------
// Every quantizer thread owns a patch of PR consecutive rows x one BYTES-wide vector
// of a row (8 bf16 / 4 fp32 for 16 bytes).  Consecutive threads take consecutive
// vectors of the same rows, so each of the PR loads is coalesced across the warp,
// and all PR loads are issued before any arithmetic (PR x BYTES bytes in flight per
// thread).  The row copy is produced row by row from the registers; the col copy
// column by column -- PR consecutive rows are exactly one column block (NVFP4: 16,
// MXFP8: 32), so no shared-memory transpose is needed.

template <typename T, int BYTES>
struct Chunk;
template <>
struct Chunk<__nv_bfloat16, 16> {
  using Raw = uint4;
  static constexpr int N = 8;
};
template <>
struct Chunk<float, 16> {
  using Raw = uint4;
  static constexpr int N = 4;
};

__device__ __forceinline__ uint4 ld_raw(const uint4* p) { return __ldg(p); }
__device__ __forceinline__ void zero_raw(uint4& r) { r = make_uint4(0, 0, 0, 0); }
__device__ __forceinline__ uint32_t raw_word(const uint4& r, int k) {
  return k == 0 ? r.x : (k == 1 ? r.y : (k == 2 ? r.z : r.w));
}
[[maybe_unused]] __device__ __forceinline__ uint32_t raw_word(const uint2& r, int k) { return k == 0 ? r.x : r.y; }

template <typename T, typename Raw>
__device__ __forceinline__ float elem(const Raw& r, int i) {
  if (sizeof(T) == 2) {
    const uint32_t w = raw_word(r, i >> 1);
    return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
  return __uint_as_float(raw_word(r, i));
}

template <typename T, int BYTES, int PR>
struct Patch {
  using Ch = Chunk<T, BYTES>;
  using Raw = typename Ch::Raw;
  static constexpr int PC = Ch::N;
  Raw raw[PR];
  int64_t r0, c0;
  bool live;

  __device__ __forceinline__ void load(const T* __restrict__ x, int64_t R, int64_t C) {
    const int64_t ncg = C / PC;
    const int64_t total = (R / PR) * ncg;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    live = idx < total;
    const int64_t band = live ? idx / ncg : 0;
    r0 = band * PR;
    c0 = live ? (idx - band * ncg) * PC : 0;
    const T* p = x + r0 * C + c0;
#pragma unroll
    for (int r = 0; r < PR; ++r) {
      if (live) raw[r] = ld_raw(reinterpret_cast<const Raw*>(p + r * C));
      else zero_raw(raw[r]);
    }
  }
  __device__ __forceinline__ float at(int r, int i) const { return elem<T>(raw[r], i); }
  __device__ __forceinline__ float absmax() const {
    float m = 0.0f;
#pragma unroll
    for (int r = 0; r < PR; ++r)
#pragma unroll
      for (int i = 0; i < PC; ++i) m = fmaxf(m, fabsf(at(r, i)));
    return m;
  }
};

inline unsigned patch_blocks(int64_t rows, int64_t cols, int pr, int pc) {
  const int64_t total = (rows / pr) * (cols / pc);
  const int64_t b = (total + kThreads - 1) / kThreads;
  return static_cast<unsigned>(b < 1 ? 1 : b);
}

// ---- amax ---------------------------------------------------------------------------------------
template <typename T, bool RHT>
__global__ void __launch_bounds__(kThreads, 2) amax_kernel(const T* __restrict__ x, int64_t R, int64_t C, float* amax,
                                                           float* amax_rht, uint32_t signs) {
  static_assert(!RHT, "the rotated amax has its own kernel");
  using P = Patch<T, 16, 16>;
  P p;
  p.load(x, R, C);
  block_max_to(p.absmax(), amax);
}

// Plain and rotated amax from one read.  Persistent grid of 3 CTAs per SM: each thread
// walks 16-row x 8-byte patches, loading one and rotating it (the other 23 warps' loads
// fill the wait; a second patch in flight per thread, at 2 CTAs per SM, was 12-15 %
// slower); columns are rotated in pairs as packed fp32 values, and the 1/4 of the
// transform is applied to the maximum (exact: scaling by 1/4 and rounding are monotone).
template <typename T, int VB, bool PLAIN>
__global__ void __launch_bounds__(kThreads, 3) amax_rht_kernel(const T* __restrict__ x, int64_t R, int64_t C,
                                                               float* amax, float* amax_rht, uint32_t signs) {
  using Vec = typename std::conditional<VB == 16, uint4, uint2>::type;
  constexpr int PC = VB / sizeof(T);   // columns per patch
  const int64_t ncg = C / PC;
  const int64_t total = (R / 16) * ncg;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  auto load = [&](int64_t i, Vec (&raw)[16]) {
    if (i < total) {
      const int64_t band = i / ncg;
      const T* q = x + band * 16 * C + (i - band * ncg) * PC;
#pragma unroll
      for (int r = 0; r < 16; ++r) raw[r] = __ldg(reinterpret_cast<const Vec*>(q + r * C));
    }
  };
  Vec cur[16];
  float m = 0.0f, mr = 0.0f;
  for (; idx < total; idx += stride) {
    load(idx, cur);
#pragma unroll
    for (int k = 0; k < PC / 2; ++k) {  // column pairs of the patch
      float2 y[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float lo, hi;
        if constexpr (sizeof(T) == 2) {
          const uint32_t w = raw_word(cur[r], k) ^ rht_sign2(signs, r);
          lo = __uint_as_float(w << 16);
          hi = __uint_as_float(w & 0xFFFF0000u);
        } else {
          const uint32_t sg = (0u - ((signs >> r) & 1u)) & 0x80000000u;
          lo = __uint_as_float(raw_word(cur[r], 2 * k) ^ sg);
          hi = __uint_as_float(raw_word(cur[r], 2 * k + 1) ^ sg);
        }
        if (PLAIN) m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
        y[r] = make_float2(lo, hi);
      }
      // Butterflies h = 1, 2, 4; the last one (h = 8) is folded into the maximum:
      // max(|fl(a + b)|, |fl(a - b)|) = fl(|a| + |b|) exactly (one of the two sums is
      // +-(|a| + |b|), the other is no larger, and rounding is symmetric and monotone).
      hadamard16x2<4>(y);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        mr = fmaxf(mr, __fadd_rn(fabsf(y[r].x), fabsf(y[r + 8].x)));
        mr = fmaxf(mr, __fadd_rn(fabsf(y[r].y), fabsf(y[r + 8].y)));
      }
    }
  }
  if (PLAIN) block_max_to(m, amax);
  block_max_to(__fmul_rn(mr, 0.25f), amax_rht);
}

// Vector width (bytes per patch row) of the rotated-amax kernel (16-byte patches need more
// registers than three CTAs per SM leave).
constexpr int kRhtAmaxVB = 8;

// ---- DelayedScaling update ----------------------------------------------------------------------
__global__ void scale_update_kernel(int n, int L, int algo, int interval, float fmax, float margin_mul,
                                    float* __restrict__ hist, const float* __restrict__ amax, float* __restrict__ scale,
                                    float* __restrict__ scale_inv, int64_t step) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float a = amax[i];
  float* h = hist + static_cast<int64_t>(i) * L;
  h[step % L] = a;
  if ((step + 1) % interval != 0) return;
  float eff = a;
  if (algo == TE_ALGO_MAX) {
    // a NaN anywhere in the window makes the maximum NaN (fmaxf would drop it), so the
    // scale is held until the NaN leaves the window, as for an infinite amax
    eff = h[0];
    for (int j = 1; j < L; ++j) {
      const float v = h[j];
      eff = (v > eff || isnan(v)) ? v : eff;
    }
  }
  float s = scale[i];
  if (isfinite(eff) && eff > 0.0f) {
    const float t = __fmul_rn(__fdiv_rn(fmax, eff), margin_mul);
    if (isfinite(t)) s = t;
  }
  scale[i] = s;
  scale_inv[i] = __fdiv_rn(1.0f, s);
}

// ---- LayerNorm fused with the FP8 cast of its output -----------------------------------------------
// Persistent CTAs of up to 12 warps (two row buffers per warp must fit in shared memory);
// each warp walks rows (grid-stride) with two shared-memory
// row buffers: lane 0 bulk-copies the next row from HBM (one cp.async.bulk per row,
// completion on the buffer's mbarrier) while the warp normalises the current one.
// Mean and biased variance are fp32 (pairs of elements as packed fp32 operations, each an
// IEEE round-to-nearest operation): each lane keeps one running sum per element position
// of its 16-byte chunks (l, l + 32, ... in order), adds the 8 sums in position order, and
// an xor-butterfly (offsets 16, 8, 4, 2, 1) combines the lanes;
// rsigma = 1 / sqrt(var + eps) (both correctly rounded).  y = fl(fl(fl(x + (-mu)) * rsigma)
// * gamma) + beta, rounded to bf16 (the LN output), and that bf16 value is cast:
// q = sat(fl32(y_bf16 * scale)); the amax of the bf16 outputs is recorded for
// DelayedScaling.
// (fl32(lo(w) + c.x), fl32(hi(w) + c.y)) for a word w of two bf16 values: the mixed-precision
// add takes the bf16 operand exactly, so this equals widening it first and adding in fp32,
// without the two instructions that widen it (LayerNorm + FP8 2-4 % faster).
__device__ __forceinline__ float2 add_bf16x2_f32(uint32_t w, float2 c) {
  float2 r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tadd.rn.f32.bf16 %0, lo, %3;\n\tadd.rn.f32.bf16 %1, hi, %4;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(w), "f"(c.x), "f"(c.y));
  return r;
}

constexpr int kLnWarps = 12;
constexpr int64_t kLnMaxCols = 8192;

__global__ void __launch_bounds__(32 * kLnWarps, 1)
    layernorm_fp8_kernel(const __nv_bfloat16* __restrict__ x, int64_t R, int64_t C, const float* __restrict__ gamma,
                         const float* __restrict__ beta, float eps, int e5m2, const float* __restrict__ scale,
                         uint8_t* __restrict__ q, __nv_bfloat16* __restrict__ ln_out, float* __restrict__ mu_out,
                         float* __restrict__ rs_out, float* amax_out, int* err) {
  extern __shared__ __align__(128) uint8_t ln_smem[];
  __shared__ uint64_t ln_bar[kLnWarps][2];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int nw = static_cast<int>(blockDim.x >> 5);   // <= kLnWarps (fewer for long rows)
  const int64_t nch = C / 8;
  const uint32_t row_bytes = static_cast<uint32_t>(C * 2);
  // gamma and beta once per CTA, then two row buffers per warp
  float4* sg = reinterpret_cast<float4*>(ln_smem);
  float4* sb = sg + C / 4;
  uint8_t* rows_base = ln_smem + C * 8;
  uint4* buf[2] = {reinterpret_cast<uint4*>(rows_base + (2 * wib) * row_bytes),
                   reinterpret_cast<uint4*>(rows_base + (2 * wib + 1) * row_bytes)};
  // gamma / beta split by chunk half: sg[h * (C / 8) + j] = gamma[8j + 4h .. 8j + 4h + 3], so the
  // lanes of a warp, which read consecutive chunks, read consecutive 16-byte words (the
  // interleaved layout put them 32 bytes apart: two-way bank conflicts; 4096 columns 8-15 % faster)
  for (int64_t i = threadIdx.x; i < C / 4; i += blockDim.x) {
    const int64_t dst = (i & 1) * (C / 8) + (i >> 1);
    sg[dst] = __ldg(reinterpret_cast<const float4*>(gamma) + i);
    sb[dst] = __ldg(reinterpret_cast<const float4*>(beta) + i);
  }
  const int64_t first = static_cast<int64_t>(blockIdx.x) * nw + wib;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * nw;
  if (lane == 0) {
    dev::mbar_init(&ln_bar[wib][0], 1);
    dev::mbar_init(&ln_bar[wib][1], 1);
    dev::fence_barrier_init();
  }
  __syncthreads();
  auto fetch = [&](int64_t row, int b) {
    dev::mbar_expect_tx(&ln_bar[wib][b], row_bytes);
    dev::bulk_load(buf[b], x + row * C, row_bytes, &ln_bar[wib][b]);
  };
  if (lane == 0 && first < R) fetch(first, 0);
  int abort_flag = 0;
  float lmax = 0.0f;
  const float sc = *scale;
  int k = 0;
  for (int64_t row = first; row < R; row += stride, ++k) {
    const int bsel = k & 1;
    if (lane == 0 && row + stride < R) fetch(row + stride, bsel ^ 1);   // that buffer's previous row is done
    // lane 0 waits for the row (bounded) and the warp follows its result together
    int ok = 1;
    if (lane == 0) ok = dev::mbar_wait(&ln_bar[wib][bsel], static_cast<uint32_t>(k >> 1) & 1u, &abort_flag, err);
    __syncwarp();
    if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
    const uint4* srow = buf[bsel];
    // per lane: 8 running sums (one per position in a chunk; pairs as packed fp32 adds),
    // added in position order
    float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    for (int64_t j = lane; j < nch; j += 32) {
      const uint4 v = srow[j];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) acc[t] = add_bf16x2_f32(w[t], acc[t]);
    }
    float sum = acc[0].x;
    sum = __fadd_rn(sum, acc[0].y);
#pragma unroll
    for (int t = 1; t < 4; ++t) sum = __fadd_rn(__fadd_rn(sum, acc[t].x), acc[t].y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, o));
    const float mu = __fdiv_rn(sum, static_cast<float>(C));
    const float2 nmu = make_float2(-mu, -mu);
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[t] = make_float2(0.f, 0.f);
    for (int64_t j = lane; j < nch; j += 32) {
      const uint4 v = srow[j];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 d = add_bf16x2_f32(w[t], nmu);
        acc[t] = __fadd2_rn(acc[t], __fmul2_rn(d, d));
      }
    }
    float sq = acc[0].x;
    sq = __fadd_rn(sq, acc[0].y);
#pragma unroll
    for (int t = 1; t < 4; ++t) sq = __fadd_rn(__fadd_rn(sq, acc[t].x), acc[t].y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xFFFFFFFFu, sq, o));
    const float var = __fdiv_rn(sq, static_cast<float>(C));
    const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
    if (lane == 0) {
      if (mu_out) mu_out[row] = mu;
      if (rs_out) rs_out[row] = rs;
    }
    const float2 rs2 = make_float2(rs, rs), sc2 = make_float2(sc, sc);
    for (int64_t j = lane; j < nch; j += 32) {
      const uint4 v = srow[j];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      const float4 g0 = sg[j], g1 = sg[C / 8 + j], b0 = sb[j], b1 = sb[C / 8 + j];
      const float2 gg[4] = {{g0.x, g0.y}, {g0.z, g0.w}, {g1.x, g1.y}, {g1.z, g1.w}};
      const float2 bb[4] = {{b0.x, b0.y}, {b0.z, b0.w}, {b1.x, b1.y}, {b1.z, b1.w}};
      uint32_t ob[4];
      float2 a[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 y = __fadd2_rn(__fmul2_rn(__fmul2_rn(add_bf16x2_f32(w[t], nmu), rs2), gg[t]), bb[t]);
        const __nv_bfloat162 yb = __floats2bfloat162_rn(y.x, y.y);   // .x in the low half
        const uint32_t bits = *reinterpret_cast<const uint32_t*>(&yb);
        ob[t] = bits;
        const float2 yv = make_float2(__uint_as_float(bits << 16), __uint_as_float(bits & 0xFFFF0000u));
        lmax = fmaxf(lmax, fmaxf(fabsf(yv.x), fabsf(yv.y)));
        a[t] = __fmul2_rn(yv, sc2);
      }
      if (ln_out) reinterpret_cast<uint4*>(ln_out + row * C)[j] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
      uint32_t qw[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint32_t lo = e5m2 ? cvt_e5m2x2(a[2 * t].x, a[2 * t].y) : cvt_e4m3x2(a[2 * t].x, a[2 * t].y);
        const uint32_t hi = e5m2 ? cvt_e5m2x2(a[2 * t + 1].x, a[2 * t + 1].y) : cvt_e4m3x2(a[2 * t + 1].x, a[2 * t + 1].y);
        qw[t] = lo | (hi << 16);
      }
      reinterpret_cast<uint2*>(q + row * C)[j] = make_uint2(qw[0], qw[1]);
    }
    __syncwarp();   // every lane is done with this buffer before lane 0 refills it
  }
  if (abort_flag && lane == 0) {
    // bounded wait for this warp's copies still in flight before the CTA exits
    int dummy = 0;
    for (int kk = k; kk < k + 2; ++kk) {
      const int64_t row = first + static_cast<int64_t>(kk) * stride;
      if (row < R) dev::mbar_wait(&ln_bar[wib][kk & 1], static_cast<uint32_t>(kk >> 1) & 1u, &dummy, err);
    }
  }
  if (amax_out != nullptr) block_max_to(lmax, amax_out);
}

// Rows of up to 4096 columns: the same arithmetic with each row held in registers (16-byte
// chunks lane, lane + 32, ...: at most 16 per lane) instead of shared-memory row buffers.
// WPR = 2 splits a row between two warps (8 chunks per lane), each warp reducing its half and
// the pair adding the two halves in a fixed order through shared memory, and holds the group's
// next row in registers as well; two CTAs of 8 warps per SM.  gamma and beta stay in shared memory.
constexpr int kLnRegCh = 16;
constexpr int64_t kLnRegMaxCols = 32 * kLnRegCh * 8;

template <int WPR>
__global__ void __launch_bounds__(256, 2)
    layernorm_fp8_reg_kernel(const __nv_bfloat16* __restrict__ x, int64_t R, int64_t C, const float* __restrict__ gamma,
                             const float* __restrict__ beta, float eps, int e5m2, const float* __restrict__ scale,
                             uint8_t* __restrict__ q, __nv_bfloat16* __restrict__ ln_out, float* __restrict__ mu_out,
                             float* __restrict__ rs_out, float* amax_out) {
  constexpr int CH = kLnRegCh / WPR;   // chunks per lane
  extern __shared__ __align__(16) float4 ln_gb[];
  __shared__ float red[8 / WPR][2][WPR];   // per row group: sum / squares partials of its warps
  float4* sg = ln_gb;
  float4* sb = ln_gb + C / 4;
  // gamma / beta split by chunk half: sg[h * (C / 8) + j] = gamma[8j + 4h .. 8j + 4h + 3], so the
  // lanes of a warp, which read consecutive chunks, read consecutive 16-byte words (the
  // interleaved layout put them 32 bytes apart: two-way bank conflicts; 4096 columns 8-15 % faster)
  for (int64_t i = threadIdx.x; i < C / 4; i += blockDim.x) {
    const int64_t dst = (i & 1) * (C / 8) + (i >> 1);
    sg[dst] = __ldg(reinterpret_cast<const float4*>(gamma) + i);
    sb[dst] = __ldg(reinterpret_cast<const float4*>(beta) + i);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int grp = wib / WPR, wr = wib % WPR;
  const int rl = wr * 32 + lane;                       // this thread's lane within its row
  const int ngrp = static_cast<int>(blockDim.x >> 5) / WPR;
  const int64_t nch = C / 8;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * ngrp + grp;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * ngrp;
  float lmax = 0.0f;
  const float sc = *scale;
  const float2 sc2 = make_float2(sc, sc);
  // the row's two warps meet at named barrier 1 + grp (64 threads)
  auto pair_sync = [&]() {
    if (WPR == 2) asm volatile("bar.sync %0, 64;" ::"r"(1 + grp) : "memory");
  };
  // row r's chunks of this lane (zeros past the row's end, or for r >= R)
  auto load_row = [&](int64_t r, uint4 (&dst)[CH]) {
    const uint4* src = reinterpret_cast<const uint4*>(x + r * C);
#pragma unroll
    for (int t = 0; t < CH; ++t) {
      const int64_t j = rl + 32 * WPR * t;
      dst[t] = (r < R && j < nch) ? __ldg(src + j) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  uint4 v[CH];
  if (WPR == 2) load_row(first, v);
  for (int64_t row = first; row < R; row += stride) {
    // WPR = 2: the group's next row is loaded while this one is normalised (1.4 % faster at
    // 4096 columns); WPR = 1 has no registers for a second row
    uint4 vn[CH];
    if (WPR == 2) load_row(row + stride, vn);
    else load_row(row, v);
    // per lane: 8 running sums (one per position in a chunk; pairs as packed fp32 adds),
    // added in position order; then an xor-butterfly over the lanes (and the row's warps)
    float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int t = 0; t < CH; ++t) {
      if (rl + 32 * WPR * t >= nch) break;
      const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] = add_bf16x2_f32(w[k], acc[k]);
    }
    float sum = acc[0].x;
    sum = __fadd_rn(sum, acc[0].y);
#pragma unroll
    for (int k = 1; k < 4; ++k) sum = __fadd_rn(__fadd_rn(sum, acc[k].x), acc[k].y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, o));
    if (WPR == 2) {
      if (lane == 0) red[grp][0][wr] = sum;
      pair_sync();
      sum = __fadd_rn(red[grp][0][0], red[grp][0][WPR - 1]);
    }
    const float mu = __fdiv_rn(sum, static_cast<float>(C));
    const float2 nmu = make_float2(-mu, -mu);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float2(0.f, 0.f);
#pragma unroll
    for (int t = 0; t < CH; ++t) {
      if (rl + 32 * WPR * t >= nch) break;
      const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 d = add_bf16x2_f32(w[k], nmu);
        acc[k] = __fadd2_rn(acc[k], __fmul2_rn(d, d));
      }
    }
    float sq = acc[0].x;
    sq = __fadd_rn(sq, acc[0].y);
#pragma unroll
    for (int k = 1; k < 4; ++k) sq = __fadd_rn(__fadd_rn(sq, acc[k].x), acc[k].y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xFFFFFFFFu, sq, o));
    if (WPR == 2) {
      if (lane == 0) red[grp][1][wr] = sq;
      pair_sync();
      sq = __fadd_rn(red[grp][1][0], red[grp][1][WPR - 1]);
    }
    const float var = __fdiv_rn(sq, static_cast<float>(C));
    const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
    if (rl == 0) {
      if (mu_out) mu_out[row] = mu;
      if (rs_out) rs_out[row] = rs;
    }
    const float2 rs2 = make_float2(rs, rs);
#pragma unroll
    for (int t = 0; t < CH; ++t) {
      const int64_t j = rl + 32 * WPR * t;
      if (j >= nch) break;
      const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
      const float4 g0 = sg[j], g1 = sg[C / 8 + j], b0 = sb[j], b1 = sb[C / 8 + j];
      const float2 gg[4] = {{g0.x, g0.y}, {g0.z, g0.w}, {g1.x, g1.y}, {g1.z, g1.w}};
      const float2 bb[4] = {{b0.x, b0.y}, {b0.z, b0.w}, {b1.x, b1.y}, {b1.z, b1.w}};
      uint32_t ob[4];
      float2 a[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 y = __fadd2_rn(__fmul2_rn(__fmul2_rn(add_bf16x2_f32(w[k], nmu), rs2), gg[k]), bb[k]);
        const __nv_bfloat162 yb = __floats2bfloat162_rn(y.x, y.y);   // .x in the low half
        const uint32_t bits = *reinterpret_cast<const uint32_t*>(&yb);
        ob[k] = bits;
        const float2 yv = make_float2(__uint_as_float(bits << 16), __uint_as_float(bits & 0xFFFF0000u));
        lmax = fmaxf(lmax, fmaxf(fabsf(yv.x), fabsf(yv.y)));
        a[k] = __fmul2_rn(yv, sc2);
      }
      if (ln_out) reinterpret_cast<uint4*>(ln_out + row * C)[j] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
      uint32_t qw[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t lo = e5m2 ? cvt_e5m2x2(a[2 * k].x, a[2 * k].y) : cvt_e4m3x2(a[2 * k].x, a[2 * k].y);
        const uint32_t hi = e5m2 ? cvt_e5m2x2(a[2 * k + 1].x, a[2 * k + 1].y) : cvt_e4m3x2(a[2 * k + 1].x, a[2 * k + 1].y);
        qw[k] = lo | (hi << 16);
      }
      reinterpret_cast<uint2*>(q + row * C)[j] = make_uint2(qw[0], qw[1]);
    }
    if (WPR == 2) {
#pragma unroll
      for (int t = 0; t < CH; ++t) v[t] = vn[t];
    }
  }
  if (amax_out != nullptr) block_max_to(lmax, amax_out);
}

// Bias gradient from the per-tile partial sums.  A CTA owns 32 columns; its 8 warps sum
// the tile rows t = w, w + 8, w + 16, ... in order, then warp 0 adds the 8 partial
// sums in warp order -- a fixed order, so the result does not depend on timing.
__global__ void __launch_bounds__(256) dbias_reduce_kernel(const float* __restrict__ ws, int64_t tiles_r, int64_t C,
                                                           float* __restrict__ dbias) {
  __shared__ float part[8][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  float s = 0.0f;
  if (c < C)
    for (int64_t t = w; t < tiles_r; t += 8) s = __fadd_rn(s, __ldg(ws + t * C + c));
  part[w][lane] = s;
  __syncthreads();
  if (w == 0 && c < C) {
    float r = part[0][lane];
#pragma unroll
    for (int k = 1; k < 8; ++k) r = __fadd_rn(r, part[k][lane]);
    dbias[c] = r;
  }
}

__device__ __forceinline__ float current_scale(float a, float fmax) {
  if (!(isfinite(a) && a > 0.0f)) return 1.0f;
  const float s = __fdiv_rn(fmax, a);
  return isfinite(s) ? s : 1.0f;
}

// Shared exponent of an MXFP8 block: clamp(floor(log2 amax) - 8, -127, 127); -127 for a zero block.
__device__ __forceinline__ int mx_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  if (b == 0) return -127;
  const uint32_t ef = b >> 23;
  int e = (ef == 0) ? (31 - __clz(static_cast<int>(b))) - 149 : static_cast<int>(ef) - 127;
  e -= 8;
  return max(-127, min(127, e));
}
__device__ __forceinline__ float mx_mult(int E) { return __uint_as_float(static_cast<uint32_t>(127 - E) << 23); }

__device__ __forceinline__ float nv_senc(float A) {
  if (!(A > 0.0f)) return 1.0f;
  const float s = __fdiv_rn(2688.0f, A);
  return isfinite(s) ? s : 1.0f;
}
// fl32(x / 6), correctly rounded, for x >= 0: the product with fl32(1/6) and one correction
// step from the exact residual (Markstein's FMA division, IBM J. Res. Dev. 34(1), 1990).  An
// exhaustive check over every float (tests/test_div6_exhaustive.py) finds it equal to the IEEE
// quotient for all x >= 2^-125; below that the quotient is subnormal and may differ by one
// ulp, so those inputs take the full division.  (Together with the RHT sign masks hoisted out
// of the block loop: NVFP4 RHT col copy 5 %, SR + RHT col copy and 2D copies 2 % faster.)
__device__ __forceinline__ float div6_rn(float x) {
  if (x >= 0x1p-125f) {
    const float c = 0x1.555556p-3f;   // fl32(1/6)
    const float q0 = __fmul_rn(x, c);
    return __fmaf_rn(__fmaf_rn(-q0, 6.0f, x), c, q0);
  }
  return __fdiv_rn(x, 6.0f);
}
// UE4M3 block-scale code of a block with amax bm: RN(fl32(fl32(bm / 6) * S_enc)).
__device__ __forceinline__ uint32_t nv_scale_code(float bm, float senc) {
  return cvt_e4m3x2(__fmul_rn(div6_rn(bm), senc), 0.0f) & 0x7Fu;
}

// ---- warp-tile quantizers (FP8, MXFP8, NVFP4) ------------------------------------------------------
// Persistent CTAs of 8 warps (NVFP4: 11, or 12 when one copy is written); every warp owns
// a private 2-stage ring of 64-row x 128-byte input tiles (64 x 64 bf16 or 64 x 32 fp32)
// that its lane 0 fills with TMA (128-byte swizzle), plus one shared-memory staging box per
// output copy written, so warps never wait on each other.  Per tile, lane l quantizes tile rows l and l + 32 for
// the row copy (16-byte shared loads, distinct swizzled chunks in every 8-lane
// phase) and its 4-byte column slice of all 64 rows for the col copy (32 distinct
// banks per row).  The quantized bytes go to swizzled staging boxes and leave with
// one TMA bulk-tensor store per copy (the hardware clips the ragged edge); block
// scales are written directly as contiguous 2-8 byte runs.

enum QFmt { kQE4M3 = 0, kQE5M2 = 1, kQMX = 2, kQNV = 3 };

struct TileArgs {
  int64_t R, C;
  int do_row, do_col;
  // per-tensor FP8
  const float* scale;
  const float* amax_in;
  int current;
  float fmax;
  float* amax_out;
  float* scale_inv_out;
  // block scales (MXFP8 / NVFP4)
  uint8_t* s_row;
  uint8_t* s_col;
  int64_t kpad_row, kpad_col;
  // NVFP4
  uint32_t flags, signs, seed_lo, seed_hi, off_lo, off_hi;
  uint32_t rk0[10], rk1[10];   // Philox round keys of (seed_lo, seed_hi)
  const float* amax;
  const float* amax_rht;
  float* gdec_row;
  float* gdec_col;
  // column sums (bias gradient): per 64-row tile, partial sums into ws[tile_row][C]
  float* dbias_ws;
  int* err;
};

constexpr int kQTileBytes = 64 * 128;   // one input tile

// 16-byte chunk j of input-tile row r (128-byte swizzle: chunk j of row r sits at j ^ (r % 8)).
__device__ __forceinline__ uint4 tile_chunk(const uint8_t* tile, int r, int j) {
  return *reinterpret_cast<const uint4*>(tile + r * 128 + ((j ^ (r & 7)) << 4));
}
// 4-byte word w (0..31) of input-tile row r.
__device__ __forceinline__ uint32_t tile_word(const uint8_t* tile, int r, int w) {
  return *reinterpret_cast<const uint32_t*>(tile + r * 128 + (((w >> 2) ^ (r & 7)) << 4) + ((w & 3) << 2));
}
// 16-byte chunk j of row r of a staging box with W-byte rows, in the TMA swizzle
// of that width (64 B: chunk ^ ((r >> 1) & 3); 32 B: chunk ^ ((r >> 2) & 1); 16 B: none).
template <int W>
__device__ __forceinline__ uint4* stage_chunk(uint8_t* box, int r, int j) {
  const int sw = W == 64 ? ((r >> 1) & 3) : (W == 32 ? ((r >> 2) & 1) : 0);
  return reinterpret_cast<uint4*>(box + r * W + ((j ^ sw) << 4));
}

template <int FMT>
__device__ __forceinline__ uint4 fp8_pack16(const float* v, float s) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float a0 = __fmul_rn(v[4 * j], s), a1 = __fmul_rn(v[4 * j + 1], s);
    const float a2 = __fmul_rn(v[4 * j + 2], s), a3 = __fmul_rn(v[4 * j + 3], s);
    const uint32_t lo = FMT == kQE5M2 ? cvt_e5m2x2(a0, a1) : cvt_e4m3x2(a0, a1);
    const uint32_t hi = FMT == kQE5M2 ? cvt_e5m2x2(a2, a3) : cvt_e4m3x2(a2, a3);
    w[j] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// 16 already-scaled NVFP4 values -> 16 E2M1 codes (element i in nibble i); with
// stochastic rounding, word i of `rnd` (one Philox output) drives elements 4i..4i+3.
template <bool SR>
__device__ __forceinline__ uint2 nv_encode16(const float* s, const uint4& rnd) {
  uint32_t lo = 0, hi = 0;
  if (!SR) {
#pragma unroll
    for (int j = 0; j < 4; ++j) lo |= cvt_e2m1x2(s[2 * j], s[2 * j + 1]) << (8 * j);
#pragma unroll
    for (int j = 0; j < 4; ++j) hi |= cvt_e2m1x2(s[8 + 2 * j], s[9 + 2 * j]) << (8 * j);
  } else {
    const uint32_t w[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = cvt_e2m1x4_rs(s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3], w[i]);
    lo = q[0] | (q[1] << 16);
    hi = q[2] | (q[3] << 16);
  }
  return make_uint2(lo, hi);
}
// 16 NVFP4 elements with their block's scale multiplier r (x * r in packed pairs).
template <bool SR>
__device__ __forceinline__ uint2 nv_pack16(const float* v, float r, const uint4& rnd) {
  const float2 rr = make_float2(r, r);
  float s[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 t = __fmul2_rn(make_float2(v[2 * i], v[2 * i + 1]), rr);
    s[2 * i] = t.x;
    s[2 * i + 1] = t.y;
  }
  return nv_encode16<SR>(s, rnd);
}

// Random words of the 16 elements g .. g + 15 (g a multiple of 16) of copy `copy_id`.
__device__ __forceinline__ uint4 nv_rand(const TileArgs& a, uint64_t g, uint32_t copy_id) {
  return philox4x32_10_rk(make_uint4(static_cast<uint32_t>(g >> 4), copy_id, a.off_lo, a.off_hi), a.rk0, a.rk1);
}

template <int L>
__device__ __forceinline__ float lanes_max(float v) {
#pragma unroll
  for (int o = 1; o < L; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// max |v_i| over 16 values with three-input maxima (8 instructions instead of 15; the
// maximum of non-negative values is exact in any order)
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float absmax16(const float (&v)[16]) {
  float m[6];
#pragma unroll
  for (int i = 0; i < 5; ++i) m[i] = max3f(fabsf(v[3 * i]), fabsf(v[3 * i + 1]), fabsf(v[3 * i + 2]));
  m[5] = fabsf(v[15]);
  return fmaxf(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]));
}

template <typename T, int FMT>
struct QGeom {
  static constexpr int TC = 128 / sizeof(T);               // tile columns
  static constexpr int NB16 = TC / 16;                     // 16-column blocks per tile row
  static constexpr int NCL = 4 / sizeof(T);                // columns per lane in the col pass
  static constexpr int ROW_W = FMT == kQNV ? TC / 2 : TC;  // staging row bytes of the row copy
  static constexpr int COL_W = FMT == kQNV ? 32 : 64;      // staging row bytes of the col copy
  static constexpr int ROW_BOX = 64 * ROW_W;               // staging box bytes of the row copy
  static constexpr int COL_BOX = TC * COL_W;               // staging box bytes of the col copy
};

// Warps per CTA and input stages per warp: 8 x 2 for FP8 / MXFP8; NVFP4, whose RHT, 2D and
// stochastic-rounding paths are latency-bound, takes 11 warps (its smaller staging boxes
// leave room): RHT col copy and 2D both copies 11-12 % faster, the RN row copy 2 % slower.
// A third stage at fewer warps, or 12 warps with one stage, were slower.
template <int FMT, bool SR>
struct QLaunch {
  static constexpr int NW = FMT == kQNV ? 11 : 8;
  static constexpr int NS = 2;
  // NVFP4 launches that write one copy leave out the other copy's staging box, which makes room
  // for a twelfth warp (SR + RHT col copy 9 % faster, RHT col 6 %, SR row 8 %); the FP8 casts
  // were slower with more warps.
  static constexpr int kOneCopyWarps = FMT == kQNV ? 12 : NW;
  static constexpr int kMaxWarps = kOneCopyWarps > NW ? kOneCopyWarps : NW;
};
template <typename T, int FMT, bool SR>
struct QSmem {
  using G = QGeom<T, FMT>;
  using Lc = QLaunch<FMT, SR>;
  static constexpr int kWarpBytes = Lc::NS * kQTileBytes + G::ROW_BOX + G::COL_BOX;
  static constexpr int kTotal = Lc::NW * kWarpBytes + 2048 /* barriers + r-tables */ + 1024 /* alignment */;
  static_assert(kTotal <= 232448, "shared memory budget");
  // one copy: the ring and that copy's box only
  static constexpr int kWarpBytesRow = Lc::NS * kQTileBytes + G::ROW_BOX;
  static constexpr int kWarpBytesCol = Lc::NS * kQTileBytes + G::COL_BOX;
  static constexpr int kTotalRow = Lc::kOneCopyWarps * kWarpBytesRow + 2048 + 1024;
  static constexpr int kTotalCol = Lc::kOneCopyWarps * kWarpBytesCol + 2048 + 1024;
  static constexpr int kTotalMax = kTotal > kTotalRow ? (kTotal > kTotalCol ? kTotal : kTotalCol)
                                                      : (kTotalRow > kTotalCol ? kTotalRow : kTotalCol);
  static_assert(kTotalMax <= 232448, "shared memory budget");
  static_assert(Lc::kMaxWarps * Lc::NS * 8 <= 256, "barrier area");
  static_assert(G::ROW_BOX % 1024 == 0 && G::COL_BOX % 1024 == 0, "box alignment");
};

// Column sums of one input tile (rows in order 0..63, fp32) for the bias gradient:
// lane l sums its 4-byte column slice (two bf16 columns or one fp32 column) and
// writes the tile row's partial sums; rows past the tensor's end were zero-filled.
template <typename T>
__device__ __forceinline__ void tile_colsum(const uint8_t* tile, int64_t r0, int64_t c0, const TileArgs& a, int lane) {
  float s0 = 0.0f, s1 = 0.0f;
#pragma unroll 16
  for (int r = 0; r < 64; ++r) {
    const uint32_t w = tile_word(tile, r, lane);
    if constexpr (sizeof(T) == 2) {
      s0 = __fadd_rn(s0, __uint_as_float(w << 16));
      s1 = __fadd_rn(s1, __uint_as_float(w & 0xFFFF0000u));
    } else {
      s0 = __fadd_rn(s0, __uint_as_float(w));
    }
  }
  constexpr int NCL = 4 / sizeof(T);
  const int64_t col = c0 + lane * NCL;
  if (col >= a.C) return;
  float* dst = a.dbias_ws + (r0 / 64) * a.C + col;
  if constexpr (sizeof(T) == 2) *reinterpret_cast<float2*>(dst) = make_float2(s0, s1);
  else *dst = s0;
}

// Row copy of one tile: lane handles rows lane and lane + 32.
template <typename T, int FMT, bool SR>
__device__ __forceinline__ void row_pass(const uint8_t* tile, uint8_t* box, int64_t r0, int64_t c0, const TileArgs& a,
                                         float s_fp8, float senc, const float* rtab, int lane, float& lmax) {
  using G = QGeom<T, FMT>;
  constexpr int NB16 = G::NB16;
  const bool two_d = FMT == kQNV && (a.flags & TE_NVFP4_2D) != 0;
  uint32_t codes[2] = {0u, 0u};  // NVFP4 / MXFP8 scale bytes of the two rows
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int rr = lane + 32 * h;
    float v[NB16][16];
#pragma unroll
    for (int j = 0; j < NB16; ++j) {
      if constexpr (sizeof(T) == 2) {
        const uint4 c0v = tile_chunk(tile, rr, 2 * j), c1v = tile_chunk(tile, rr, 2 * j + 1);
        const uint32_t w[8] = {c0v.x, c0v.y, c0v.z, c0v.w, c1v.x, c1v.y, c1v.z, c1v.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[j][2 * i] = __uint_as_float(w[i] << 16);
          v[j][2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 c = tile_chunk(tile, rr, 4 * j + q);
          v[j][4 * q] = __uint_as_float(c.x);
          v[j][4 * q + 1] = __uint_as_float(c.y);
          v[j][4 * q + 2] = __uint_as_float(c.z);
          v[j][4 * q + 3] = __uint_as_float(c.w);
        }
      }
    }
    float bmax[NB16];
#pragma unroll
    for (int j = 0; j < NB16; ++j) {
      const float m = absmax16(v[j]);
      bmax[j] = m;
      lmax = fmaxf(lmax, m);
    }
    if constexpr (FMT == kQE4M3 || FMT == kQE5M2) {
#pragma unroll
      for (int j = 0; j < NB16; ++j) *stage_chunk<G::ROW_W>(box, rr, j) = fp8_pack16<FMT>(v[j], s_fp8);
    } else if constexpr (FMT == kQMX) {
#pragma unroll
      for (int j = 0; j < NB16; j += 2) {
        const int E = mx_exponent(fmaxf(bmax[j], bmax[j + 1]));
        const float mult = mx_mult(E);
        *stage_chunk<G::ROW_W>(box, rr, j) = fp8_pack16<kQE4M3>(v[j], mult);
        *stage_chunk<G::ROW_W>(box, rr, j + 1) = fp8_pack16<kQE4M3>(v[j + 1], mult);
        codes[h] |= static_cast<uint32_t>(E + 127) << (8 * (j / 2));
      }
    } else {
      if (two_d) {
#pragma unroll
        for (int j = 0; j < NB16; ++j) bmax[j] = lanes_max<16>(bmax[j]);  // 16 rows x 16 cols
      }
      const uint64_t g = static_cast<uint64_t>(r0 + rr) * static_cast<uint64_t>(a.C) + static_cast<uint64_t>(c0);
      uint2 q[NB16];
#pragma unroll
      for (int j = 0; j < NB16; ++j) {
        const uint32_t sc = nv_scale_code(bmax[j], senc);
        codes[h] |= sc << (8 * j);
        uint4 rnd = make_uint4(0, 0, 0, 0);
        if (SR) rnd = nv_rand(a, g + 16 * j, 0u);
        q[j] = nv_pack16<SR>(v[j], rtab[sc], rnd);
      }
#pragma unroll
      for (int j = 0; j < NB16; j += 2)
        *stage_chunk<G::ROW_W>(box, rr, j / 2) = make_uint4(q[j].x, q[j].y, q[j + 1].x, q[j + 1].y);
    }
  }
  if constexpr (FMT == kQNV || FMT == kQMX) {
    // rows r0 + lane and r0 + lane + 32 share a 16-byte row of the scale atom, 4 bytes apart
    const int64_t row = r0 + lane;
    if (row < a.R) {
      const int64_t jb = FMT == kQNV ? c0 / 16 : c0 / 32;
      uint8_t* dst = a.s_row + scale_offset(row, jb, a.kpad_row);
      const bool both = row + 32 < a.R;
      if constexpr (FMT == kQNV && NB16 == 4) {
        if (both) *reinterpret_cast<uint2*>(dst) = make_uint2(codes[0], codes[1]);
        else *reinterpret_cast<uint32_t*>(dst) = codes[0];
      } else if constexpr (FMT == kQNV || (FMT == kQMX && NB16 == 4)) {   // 2 scale bytes per row
        *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(codes[0]);
        if (both) *reinterpret_cast<uint16_t*>(dst + 4) = static_cast<uint16_t>(codes[1]);
      } else {                                                            // 1 scale byte per row
        dst[0] = static_cast<uint8_t>(codes[0]);
        if (both) dst[4] = static_cast<uint8_t>(codes[1]);
      }
    }
  }
}

// Col copy of one tile: lane handles its 4-byte column slice (NCL columns) of all 64 rows.
template <typename T, int FMT, bool SR>
// smask[r]: the RHT sign-flip mask of block row r (zero without RHT), computed once per kernel.
__device__ __forceinline__ void col_pass(const uint8_t* tile, uint8_t* box, int64_t r0, int64_t c0, const TileArgs& a,
                                         float s_fp8, float senc, const float* rtab, int lane, float& lmax,
                                         bool track_max, const uint32_t (&smask)[16]) {
  using G = QGeom<T, FMT>;
  constexpr int NCL = G::NCL;
  const bool two_d = FMT == kQNV && (a.flags & TE_NVFP4_2D) != 0;
  const bool rht = FMT == kQNV && (a.flags & TE_NVFP4_RHT_COL) != 0;
  uint32_t codes[NCL] = {};
  constexpr int RB = FMT == kQMX ? 32 : 16;  // rows per block of the col copy
  if constexpr (FMT == kQNV && NCL == 2) {
    // NVFP4, two columns per lane: both columns travel as packed fp32 pairs
    // through the sign flip, the Hadamard butterflies, the 1/4 and the block scaling.
    // all four 16-row blocks of the tile in flight (stochastic rounding: 3 % faster than two)
    uint2 qa_all[4], qb_all[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      // The block's random words depend only on its position: drawn first, so that the
      // generator's dependent rounds overlap the loads and the butterflies below.
      uint4 rnd_a = make_uint4(0, 0, 0, 0), rnd_b = rnd_a;
      if (SR) {
        const uint64_t g = static_cast<uint64_t>(c0 + 2 * lane) * static_cast<uint64_t>(a.R) +
                           static_cast<uint64_t>(r0 + b * 16);
        rnd_a = nv_rand(a, g, 1u);
        rnd_b = nv_rand(a, g + static_cast<uint64_t>(a.R), 1u);
      }
      float2 y[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        uint32_t w = tile_word(tile, b * 16 + r, lane);
        w ^= smask[r];
        y[r] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
      }
      if (rht) {
        hadamard16x2(y);
#pragma unroll
        for (int r = 0; r < 16; ++r) y[r] = __fmul2_rn(y[r], make_float2(0.25f, 0.25f));
      }
      float ta[16], tb[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) ta[r] = y[r].x, tb[r] = y[r].y;
      float ma = absmax16(ta), mb = absmax16(tb);
      if (two_d) ma = mb = lanes_max<8>(fmaxf(ma, mb));  // 16 rows x 16 columns
      const uint32_t sa = nv_scale_code(ma, senc), sb = nv_scale_code(mb, senc);
      codes[0] |= sa << (8 * b);
      codes[1] |= sb << (8 * b);
      const float2 rr = make_float2(rtab[sa], rtab[sb]);
      float va[16], vb[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const float2 t = __fmul2_rn(y[r], rr);
        va[r] = t.x;
        vb[r] = t.y;
      }
      qa_all[b] = nv_encode16<SR>(va, rnd_a);
      qb_all[b] = nv_encode16<SR>(vb, rnd_b);
      // Two blocks fill one 16-byte chunk of each 32-byte box row.  Whole chunks, not 8-byte
      // halves, are stored: lanes 64 bytes apart made the halves 8-way bank conflicts.  With
      // stochastic rounding a chunk goes out as soon as its two blocks are done, without it at
      // the end of the tile (SR + RHT col copy 5.5 %, RHT col copy 5.6 % faster than 8-byte halves).
      if (SR && (b & 1)) {
        *stage_chunk<G::COL_W>(box, 2 * lane, b >> 1) = make_uint4(qa_all[b - 1].x, qa_all[b - 1].y, qa_all[b].x, qa_all[b].y);
        *stage_chunk<G::COL_W>(box, 2 * lane + 1, b >> 1) =
            make_uint4(qb_all[b - 1].x, qb_all[b - 1].y, qb_all[b].x, qb_all[b].y);
      }
    }
    if (!SR) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        *stage_chunk<G::COL_W>(box, 2 * lane, h) = make_uint4(qa_all[2 * h].x, qa_all[2 * h].y, qa_all[2 * h + 1].x, qa_all[2 * h + 1].y);
        *stage_chunk<G::COL_W>(box, 2 * lane + 1, h) =
            make_uint4(qb_all[2 * h].x, qb_all[2 * h].y, qb_all[2 * h + 1].x, qb_all[2 * h + 1].y);
      }
    }
  } else {
#pragma unroll 1
    for (int b = 0; b < 64 / RB; ++b) {
      float v[NCL][RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const uint32_t w = tile_word(tile, b * RB + r, lane);
        if constexpr (sizeof(T) == 2) {
          v[0][r] = __uint_as_float(w << 16);
          v[NCL - 1][r] = __uint_as_float(w & 0xFFFF0000u);
        } else {
          v[0][r] = __uint_as_float(w);
        }
      }
      float tile_m = 0.0f;
      if (two_d) {
#pragma unroll
        for (int qq = 0; qq < NCL; ++qq)
#pragma unroll
          for (int r = 0; r < RB; ++r) tile_m = fmaxf(tile_m, fabsf(v[qq][r]));
        tile_m = lanes_max<16 / NCL>(tile_m);  // 16 rows x 16 columns
      }
#pragma unroll
      for (int q = 0; q < NCL; ++q) {
        const int cl = lane * NCL + q;  // column within the tile = row of the col-copy box
        if constexpr (FMT == kQE4M3 || FMT == kQE5M2) {
          if (track_max)
#pragma unroll
            for (int r = 0; r < RB; ++r) lmax = fmaxf(lmax, fabsf(v[q][r]));
          *stage_chunk<G::COL_W>(box, cl, b) = fp8_pack16<FMT>(v[q], s_fp8);
        } else if constexpr (FMT == kQMX) {
          float m = 0.0f;
#pragma unroll
          for (int r = 0; r < RB; ++r) m = fmaxf(m, fabsf(v[q][r]));
          const int E = mx_exponent(m);
          const float mult = mx_mult(E);
          *stage_chunk<G::COL_W>(box, cl, 2 * b) = fp8_pack16<kQE4M3>(&v[q][0], mult);
          *stage_chunk<G::COL_W>(box, cl, 2 * b + 1) = fp8_pack16<kQE4M3>(&v[q][16], mult);
          codes[q] |= static_cast<uint32_t>(E + 127) << (8 * b);
        } else {
          float x[16];
#pragma unroll
          for (int r = 0; r < 16; ++r) x[r] = v[q][r];
          if (rht) rht16(x, a.signs);
          float m = tile_m;
          if (!two_d) {
            m = 0.0f;
#pragma unroll
            for (int r = 0; r < 16; ++r) m = fmaxf(m, fabsf(x[r]));
          }
          const uint32_t sc = nv_scale_code(m, senc);
          codes[q] |= sc << (8 * b);
          uint4 rnd = make_uint4(0, 0, 0, 0);
          if (SR)
            rnd = nv_rand(a, static_cast<uint64_t>(c0 + cl) * static_cast<uint64_t>(a.R) + static_cast<uint64_t>(r0 + b * 16),
                          1u);
          const uint2 qv = nv_pack16<SR>(x, rtab[sc], rnd);
          // two 16-row blocks share one 16-byte chunk of the 32-byte box row
          uint8_t* dst = reinterpret_cast<uint8_t*>(stage_chunk<G::COL_W>(box, cl, b >> 1)) + (b & 1) * 8;
          *reinterpret_cast<uint2*>(dst) = qv;
        }
      }
    }
  }
  if constexpr (FMT == kQNV || FMT == kQMX) {
#pragma unroll
    for (int q = 0; q < NCL; ++q) {
      const int64_t col = c0 + lane * NCL + q;
      if (col < a.C) {
        uint8_t* dst = a.s_col + scale_offset(col, FMT == kQNV ? r0 / 16 : r0 / 32, a.kpad_col);
        if constexpr (FMT == kQNV) *reinterpret_cast<uint32_t*>(dst) = codes[q];
        else *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(codes[q]);
      }
    }
  }
}

template <typename T, int FMT, bool SR>
__global__ void __launch_bounds__(QLaunch<FMT, SR>::kMaxWarps * 32, 1)
    qtile_kernel(const __grid_constant__ CUtensorMap tm_in, const __grid_constant__ CUtensorMap tm_row,
                 const __grid_constant__ CUtensorMap tm_col, const __grid_constant__ TileArgs a) {
  using G = QGeom<T, FMT>;
  constexpr int TC = G::TC;
  using Sm = QSmem<T, FMT, SR>;
  using Lc = QLaunch<FMT, SR>;
  // NVFP4 one-copy launches carry more warps, each with the input ring and that copy's box only
  const bool one_copy = Lc::kOneCopyWarps != Lc::NW && !(a.do_row && a.do_col);
  const int kQWarps = Lc::kOneCopyWarps != Lc::NW ? static_cast<int>(blockDim.x >> 5) : Lc::NW;
  constexpr int kQStages = Lc::NS;
  const int kQWarpBytes = one_copy ? (a.do_row ? Sm::kWarpBytesRow : Sm::kWarpBytesCol) : Sm::kWarpBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = dev::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + warp * kQWarpBytes;
  uint8_t* box_row = ring + kQStages * kQTileBytes;
  uint8_t* box_col = box_row + (one_copy && !a.do_row ? 0 : G::ROW_BOX);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kQWarps * kQWarpBytes) + warp * kQStages;
  float* rtab = reinterpret_cast<float*>(smem + kQWarps * kQWarpBytes + 256);

  float s_fp8 = 1.0f, senc_r = 1.0f, senc_c = 1.0f;
  if (FMT == kQE4M3 || FMT == kQE5M2) s_fp8 = a.current ? current_scale(*a.amax_in, a.fmax) : *a.scale;
  if (FMT == kQNV) {
    const bool rht = (a.flags & TE_NVFP4_RHT_COL) != 0;
    if (a.do_row) senc_r = nv_senc(*a.amax);
    if (a.do_col) senc_c = nv_senc(rht ? *a.amax_rht : *a.amax);
    if (threadIdx.x < 128) {
      const float dv = ue4m3_value(threadIdx.x);
      rtab[threadIdx.x] = dv > 0.0f ? __fdiv_rn(senc_r, dv) : 0.0f;
      rtab[128 + threadIdx.x] = dv > 0.0f ? __fdiv_rn(senc_c, dv) : 0.0f;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      if (a.gdec_row != nullptr) *a.gdec_row = __fdiv_rn(1.0f, senc_r);
      if (a.gdec_col != nullptr) *a.gdec_col = __fdiv_rn(1.0f, senc_c);
    }
  }
  if ((FMT == kQE4M3 || FMT == kQE5M2) && a.scale_inv_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0)
    *a.scale_inv_out = __fdiv_rn(1.0f, s_fp8);
  if (lane == 0) {
    for (int s = 0; s < kQStages; ++s) dev::mbar_init(&bars[s], 1);
    dev::fence_barrier_init();
  }
  __syncthreads();

  const int64_t tiles_c = (a.C + TC - 1) / TC;
  const int64_t n = ((a.R + 63) / 64) * tiles_c;
  const int64_t W = static_cast<int64_t>(gridDim.x) * kQWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kQWarps + warp;
  // Work item t covers tile n - 1 - t: the tensor is walked from its end backwards, so
  // that the tiles an amax pass over the same tensor read last (forwards, just before
  // this launch) are the first ones read here, while they are still in L2.
  const int64_t last = n - 1;
  if (lane == 0) {
    for (int s = 0; s < kQStages; ++s) {
      const int64_t t = first + s * W;
      if (t < n) {
        dev::mbar_expect_tx(&bars[s], kQTileBytes);
        dev::tma_load_2d(ring + s * kQTileBytes, &tm_in, &bars[s], static_cast<int>(((last - t) % tiles_c) * 128),
                         static_cast<int>(((last - t) / tiles_c) * 64));
      }
    }
  }
  // the 16 RHT sign masks of a block's rows, once per kernel instead of once per block
  uint32_t smask[16];
  const bool rht_col = FMT == kQNV && (a.flags & TE_NVFP4_RHT_COL) != 0;
#pragma unroll
  for (int r = 0; r < 16; ++r) smask[r] = rht_col ? rht_sign2(a.signs, r) : 0u;
  int abort_flag = 0;
  float lmax = 0.0f;
  int k = 0;
  for (int64_t t = first; t < n; t += W, ++k) {
    const int s = k % kQStages;
    const uint32_t ph = static_cast<uint32_t>(k / kQStages) & 1u;
    if (!dev::mbar_wait(&bars[s], ph, &abort_flag, a.err)) break;
    const int64_t r0 = ((last - t) / tiles_c) * 64, c0 = ((last - t) % tiles_c) * TC;
    const uint8_t* tile = ring + s * kQTileBytes;
    if (lane == 0) dev::bulk_wait_read0();  // the previous tile's boxes have been read out
    __syncwarp();
    if (a.do_row) row_pass<T, FMT, SR>(tile, box_row, r0, c0, a, s_fp8, senc_r, rtab, lane, lmax);
    if (a.do_col) col_pass<T, FMT, SR>(tile, box_col, r0, c0, a, s_fp8, senc_c, rtab + 128, lane, lmax, !a.do_row, smask);
    if (a.dbias_ws != nullptr) tile_colsum<T>(tile, r0, c0, a, lane);
    dev::fence_proxy_async();  // order this tile's shared-memory reads and box writes before the async copies
    __syncwarp();
    if (lane == 0) {
      if (a.do_row) dev::tma_store_2d(&tm_row, box_row, static_cast<int>(c0 * G::ROW_W / TC), static_cast<int>(r0));
      if (a.do_col) dev::tma_store_2d(&tm_col, box_col, static_cast<int>(r0 * G::COL_W / 64), static_cast<int>(c0));
      dev::bulk_commit();
      const int64_t nt = t + kQStages * W;
      if (nt < n) {
        dev::mbar_expect_tx(&bars[s], kQTileBytes);
        dev::tma_load_2d(ring + s * kQTileBytes, &tm_in, &bars[s], static_cast<int>(((last - nt) % tiles_c) * 128),
                         static_cast<int>(((last - nt) / tiles_c) * 64));
      }
    }
  }
  if (abort_flag) {
    // bounded wait for this warp's own loads still in flight before the CTA exits
    int dummy = 0;
    for (int j = 0; j < kQStages; ++j) {
      const int kk = k + j;
      const int64_t t = first + static_cast<int64_t>(kk) * W;
      if (t < n) dev::mbar_wait(&bars[kk % kQStages], static_cast<uint32_t>(kk / kQStages) & 1u, &dummy, a.err);
    }
  }
  if (lane == 0) dev::bulk_wait0();
  if ((FMT == kQE4M3 || FMT == kQE5M2) && a.amax_out != nullptr) {
    lmax = warp_max(lmax);
    if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(a.amax_out), __float_as_uint(lmax));
  }
}

// ---- host helpers ----------------------------------------------------------------------------------

inline bool in_dtype_ok(te_dtype d) { return d == TE_BF16 || d == TE_F32; }

inline te_status check_2d(const void* x, te_dtype in, int64_t rows, int64_t cols) {
  if (!in_dtype_ok(in)) return TE_ERR_DTYPE;
  if (rows < 0 || cols < 0 || rows % 16 || cols % 16) return TE_ERR_SHAPE;
  if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31)) return TE_ERR_SHAPE;
  // patches are counted with 64-bit indices; keep the grid within 2^31 blocks and
  // element indices of the stochastic-rounding counters below 2^34
  if (rows * cols >= (int64_t(1) << 34)) return TE_ERR_SHAPE;
  if (rows * cols > 0) {
    if (x == nullptr) return TE_ERR_NULL;
    if (!aligned16(x)) return TE_ERR_ALIGN;
  }
  return TE_OK;
}

te_status launch_amax(const void* x, te_dtype in, int64_t rows, int64_t cols, float* amax, float* amax_rht,
                      uint32_t signs, cudaStream_t st) {
  if (amax != nullptr && cudaMemsetAsync(amax, 0, sizeof(float), st) != cudaSuccess)
    return record_cuda(cudaGetLastError());
  if (amax_rht != nullptr && cudaMemsetAsync(amax_rht, 0, sizeof(float), st) != cudaSuccess)
    return record_cuda(cudaGetLastError());
  if (rows * cols == 0) return TE_OK;
  if (amax_rht != nullptr) {
    const int64_t patches = (rows / 16) * (cols / (in == TE_BF16 ? kRhtAmaxVB / 2 : kRhtAmaxVB / 4));
    const int64_t want = (patches + kThreads - 1) / kThreads;
    const unsigned grid = static_cast<unsigned>(want < 3 * num_sms() ? want : 3 * num_sms());
    if (in == TE_BF16) {
      auto* p = static_cast<const __nv_bfloat16*>(x);
      if (amax != nullptr)
        amax_rht_kernel<__nv_bfloat16, kRhtAmaxVB, true><<<grid, kThreads, 0, st>>>(p, rows, cols, amax, amax_rht,
                                                                                    signs);
      else
        amax_rht_kernel<__nv_bfloat16, kRhtAmaxVB, false><<<grid, kThreads, 0, st>>>(p, rows, cols, amax, amax_rht,
                                                                                     signs);
    } else {
      auto* p = static_cast<const float*>(x);
      if (amax != nullptr)
        amax_rht_kernel<float, kRhtAmaxVB, true><<<grid, kThreads, 0, st>>>(p, rows, cols, amax, amax_rht, signs);
      else
        amax_rht_kernel<float, kRhtAmaxVB, false><<<grid, kThreads, 0, st>>>(p, rows, cols, amax, amax_rht, signs);
    }
  } else if (in == TE_BF16) {
    amax_kernel<__nv_bfloat16, false><<<patch_blocks(rows, cols, 16, 8), kThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), rows, cols, amax, nullptr, signs);
  } else {
    amax_kernel<float, false><<<patch_blocks(rows, cols, 16, 4), kThreads, 0, st>>>(static_cast<const float*>(x), rows,
                                                                                 cols, amax, nullptr, signs);
  }
  count_launch();
  return launch_status();
}

te_status zero_scales(uint8_t* s, te_dtype fmt, int64_t rows, int64_t cols, cudaStream_t st) {
  const int64_t blk = fmt == TE_E8M0 ? 32 : 16;
  const size_t bytes = te_scale_bytes(fmt, rows, cols);
  const bool padded = (rows % 128) != 0 || ((cols / blk) % (fmt == TE_E8M0 ? 4 : 16)) != 0;
  if (padded && bytes > 0 && cudaMemsetAsync(s, 0, bytes, st) != cudaSuccess) return record_cuda(cudaGetLastError());
  return TE_OK;
}

inline int64_t kpad_of(te_dtype fmt, int64_t cols) {
  return fmt == TE_E8M0 ? ((cols / 32 + 3) / 4) * 4 : ((cols / 16 + 15) / 16) * 16;
}


template <typename T, int FMT, bool SR>
te_status launch_qtile(const void* x, int64_t R, int64_t C, uint8_t* q_row, uint8_t* q_col, TileArgs a,
                       cudaStream_t st) {
  using G = QGeom<T, FMT>;
  static bool attr_set[64] = {false};
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  if (dev_id >= 0 && dev_id < 64 && !attr_set[dev_id]) {
    if (cudaFuncSetAttribute(qtile_kernel<T, FMT, SR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             QSmem<T, FMT, SR>::kTotalMax) != cudaSuccess)
      return record_cuda(cudaGetLastError());
    attr_set[dev_id] = true;
  }
  CUtensorMap tin, trow, tcol;
  memset(&tin, 0, sizeof(tin));
  memset(&trow, 0, sizeof(trow));
  memset(&tcol, 0, sizeof(tcol));
  a.do_row = q_row != nullptr;
  a.do_col = q_col != nullptr;
  if (R * C > 0) {
    te_status s = make_tmap_2d(&tin, x, static_cast<uint64_t>(C) * sizeof(T), static_cast<uint64_t>(R), 64);
    if (s == TE_OK && q_row)
      s = make_tmap_2d_boxswz(&trow, q_row, static_cast<uint64_t>(FMT == kQNV ? C / 2 : C), static_cast<uint64_t>(R),
                              G::ROW_W, 64);
    if (s == TE_OK && q_col)
      s = make_tmap_2d_boxswz(&tcol, q_col, static_cast<uint64_t>(FMT == kQNV ? R / 2 : R), static_cast<uint64_t>(C),
                              G::COL_W, G::TC);
    if (s != TE_OK) return s;
  }
  a.err = device_error_word();
  if (a.err == nullptr) return record_cuda(cudaErrorInvalidDevice);
  constexpr int TC = G::TC;
  using Sm = QSmem<T, FMT, SR>;
  const bool one_copy = QLaunch<FMT, SR>::kOneCopyWarps != QLaunch<FMT, SR>::NW && (q_row == nullptr || q_col == nullptr);
  const int NW = one_copy ? QLaunch<FMT, SR>::kOneCopyWarps : QLaunch<FMT, SR>::NW;
  const int smem_bytes = one_copy ? (q_row ? Sm::kTotalRow : Sm::kTotalCol) : Sm::kTotal;
  const int64_t tiles = ((R + 63) / 64) * ((C + TC - 1) / TC);
  int64_t grid = (tiles + NW - 1) / NW;
  if (grid > num_sms()) grid = num_sms();
  if (grid < 1) grid = 1;
  qtile_kernel<T, FMT, SR><<<static_cast<unsigned>(grid), NW * 32, smem_bytes, st>>>(tin, trow, tcol, a);
  count_launch();
  return launch_status();
}

template <int FMT, bool SR>
te_status launch_qtile_any(const void* x, te_dtype in, int64_t R, int64_t C, uint8_t* q_row, uint8_t* q_col,
                           const TileArgs& a, cudaStream_t st) {
  if (in == TE_BF16) return launch_qtile<__nv_bfloat16, FMT, SR>(x, R, C, q_row, q_col, a, st);
  return launch_qtile<float, FMT, SR>(x, R, C, q_row, q_col, a, st);
}

}  // namespace
}  // namespace te

using namespace te;

extern "C" {

te_status te_amax_reduce(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, float* amax, float* amax_rht,
                         uint32_t rht_signs, void* stream) {
  te_status s = check_2d(x, in_dtype, rows, cols);
  if (s != TE_OK) return s;
  if (amax == nullptr && amax_rht == nullptr) return TE_ERR_NULL;
  return launch_amax(x, in_dtype, rows, cols, amax, amax_rht, rht_signs & 0xFFFFu, static_cast<cudaStream_t>(stream));
}

te_status te_scale_update(const te_recipe* recipe, int is_backward, int n_tensors, float* hist, const float* amax,
                          float* scale, float* scale_inv, int64_t step, void* stream) {
  if (recipe == nullptr) return TE_ERR_NULL;
  const te_dtype fmt = is_backward ? recipe->bwd_fmt : recipe->fwd_fmt;
  if (fmt != TE_E4M3 && fmt != TE_E5M2) return TE_ERR_DTYPE;
  if (recipe->amax_history_len < 1 || recipe->interval < 1 || recipe->margin < 0 || recipe->margin > 64 ||
      (recipe->amax_compute_algo != TE_ALGO_MAX && recipe->amax_compute_algo != TE_ALGO_MOST_RECENT) || step < 0 ||
      n_tensors < 0)
    return TE_ERR_ARG;
  if (n_tensors == 0) return TE_OK;
  if (!hist || !amax || !scale || !scale_inv) return TE_ERR_NULL;
  const float fmax = fmt == TE_E4M3 ? 448.0f : 57344.0f;
  const uint32_t mbits = static_cast<uint32_t>(127 - recipe->margin) << 23;  // 2^-margin, exact
  float margin_mul;
  memcpy(&margin_mul, &mbits, sizeof(float));
  const int threads = 128;
  scale_update_kernel<<<(n_tensors + threads - 1) / threads, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      n_tensors, recipe->amax_history_len, recipe->amax_compute_algo, recipe->interval, fmax, margin_mul, hist, amax,
      scale, scale_inv, step);
  count_launch();
  return launch_status();
}

size_t te_dbias_workspace_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return 0;
  return static_cast<size_t>((rows + 63) / 64) * static_cast<size_t>(cols) * sizeof(float);
}

}  // extern "C"

namespace {
// Host-side checks of the per-tensor FP8 cast's arguments (everything but the dbias workspace).
te_status check_fp8_cast(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, te_dtype fmt,
                         const float* scale, int compute_scale, const uint8_t* q_row, const uint8_t* q_col,
                         const float* amax_out, const float* dbias) {
  te_status s = check_2d(x, in_dtype, rows, cols);
  if (s != TE_OK) return s;
  if (fmt != TE_E4M3 && fmt != TE_E5M2) return TE_ERR_DTYPE;
  if (compute_scale != 0 && compute_scale != 1) return TE_ERR_ARG;
  if (compute_scale ? amax_out == nullptr : scale == nullptr) return TE_ERR_NULL;
  if ((q_row && !aligned16(q_row)) || (q_col && !aligned16(q_col))) return TE_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(dbias) & 3u) return TE_ERR_ALIGN;
  return TE_OK;
}
}  // namespace

extern "C" {

te_status te_quantize_fp8_dbias(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, te_dtype fmt,
                                const float* scale, int compute_scale, uint8_t* q_row, uint8_t* q_col, float* amax_out,
                                float* scale_inv_out, float* dbias, float* workspace, size_t workspace_bytes,
                                void* stream) {
  te_status s = check_fp8_cast(x, in_dtype, rows, cols, fmt, scale, compute_scale, q_row, q_col, amax_out, dbias);
  if (s != TE_OK) return s;
  const bool want_dbias = dbias != nullptr;
  if (want_dbias && cols > 0) {
    if (rows > 0 && workspace == nullptr) return TE_ERR_NULL;
    if (rows > 0 && workspace_bytes < te_dbias_workspace_bytes(rows, cols)) return TE_ERR_SHAPE;
    if ((rows > 0 && !aligned16(workspace)) || (reinterpret_cast<uintptr_t>(dbias) & 3u)) return TE_ERR_ALIGN;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (compute_scale) {
    s = launch_amax(x, in_dtype, rows, cols, amax_out, nullptr, 0, st);
    if (s != TE_OK) return s;
  } else if (amax_out != nullptr) {
    if (cudaMemsetAsync(amax_out, 0, sizeof(float), st) != cudaSuccess) return record_cuda(cudaGetLastError());
  }
  if (want_dbias && rows == 0 && cols > 0) {
    if (cudaMemsetAsync(dbias, 0, static_cast<size_t>(cols) * sizeof(float), st) != cudaSuccess)
      return record_cuda(cudaGetLastError());
  }
  if (rows * cols == 0 && scale_inv_out == nullptr) return TE_OK;
  // An empty tensor still launches one (load-free) CTA so that scale_inv_out is published.
  TileArgs a{};
  a.R = rows;
  a.C = cols;
  a.scale = scale;
  a.amax_in = amax_out;
  a.current = compute_scale;
  a.fmax = fmt == TE_E4M3 ? 448.0f : 57344.0f;
  a.amax_out = compute_scale ? nullptr : amax_out;
  a.scale_inv_out = scale_inv_out;
  a.dbias_ws = (want_dbias && rows * cols > 0) ? workspace : nullptr;
  s = fmt == TE_E4M3 ? launch_qtile_any<kQE4M3, false>(x, in_dtype, rows, cols, q_row, q_col, a, st)
                     : launch_qtile_any<kQE5M2, false>(x, in_dtype, rows, cols, q_row, q_col, a, st);
  if (s != TE_OK || a.dbias_ws == nullptr) return s;
  const int64_t tiles_r = (rows + 63) / 64;
  dbias_reduce_kernel<<<static_cast<unsigned>((cols + 31) / 32), 256, 0, st>>>(workspace, tiles_r, cols, dbias);
  count_launch();
  return launch_status();
}

te_status te_quantize_fp8(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, te_dtype fmt,
                          const float* scale, int compute_scale, uint8_t* q_row, uint8_t* q_col, float* amax_out,
                          float* scale_inv_out, void* stream) {
  return te_quantize_fp8_dbias(x, in_dtype, rows, cols, fmt, scale, compute_scale, q_row, q_col, amax_out,
                               scale_inv_out, nullptr, nullptr, 0, stream);
}

te_status te_layernorm_fp8(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, const float* gamma,
                           const float* beta, float eps, te_dtype fmt, const float* scale, uint8_t* q_row,
                           void* ln_out, float* mu, float* rsigma, float* amax_out, float* scale_inv_out,
                           void* stream) {
  te_status s = check_2d(x, in_dtype, rows, cols);
  if (s != TE_OK) return s;
  if (in_dtype != TE_BF16 || (fmt != TE_E4M3 && fmt != TE_E5M2)) return TE_ERR_DTYPE;
  if (cols % 16 != 0 || cols > kLnMaxCols) return TE_ERR_SHAPE;
  if (!(eps >= 0.0f) || !isfinite(eps)) return TE_ERR_ARG;
  if (scale == nullptr || q_row == nullptr || gamma == nullptr || beta == nullptr) return TE_ERR_NULL;
  if (!aligned16(q_row) || !aligned16(gamma) || !aligned16(beta) || (ln_out && !aligned16(ln_out)))
    return TE_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (amax_out != nullptr && cudaMemsetAsync(amax_out, 0, sizeof(float), st) != cudaSuccess)
    return record_cuda(cudaGetLastError());
  if (rows > 0 && cols <= kLnRegMaxCols) {
    // two warps per row above 2048 columns (4096: 3 % faster), one below (768-1024: 7 % faster)
    const int wpr = cols > 2048 ? 2 : 1;
    const int64_t rows_per_cta = 8 / wpr, ctas_per_sm = 2;
    const int64_t want = (rows + rows_per_cta - 1) / rows_per_cta;
    const unsigned grid = static_cast<unsigned>(want < ctas_per_sm * num_sms() ? want : ctas_per_sm * num_sms());
    auto* xp = static_cast<const __nv_bfloat16*>(x);
    auto* lp = static_cast<__nv_bfloat16*>(ln_out);
    if (wpr == 2)
      layernorm_fp8_reg_kernel<2><<<grid, 256, static_cast<size_t>(8 * cols), st>>>(
          xp, rows, cols, gamma, beta, eps, fmt == TE_E5M2, scale, q_row, lp, mu, rsigma, amax_out);
    else
      layernorm_fp8_reg_kernel<1><<<grid, 256, static_cast<size_t>(8 * cols), st>>>(
          xp, rows, cols, gamma, beta, eps, fmt == TE_E5M2, scale, q_row, lp, mu, rsigma, amax_out);
    count_launch();
    s = launch_status();
    if (s != TE_OK) return s;
  } else if (rows > 0) {
    // gamma, beta (8 B per column) and two bf16 row buffers per warp within 224 KB
    const int64_t fit = (224 * 1024 - 8 * cols) / (4 * cols);
    const int nw = static_cast<int>(fit < kLnWarps ? fit : kLnWarps);
    const size_t smem = static_cast<size_t>(8 * cols) + static_cast<size_t>(2 * nw) * static_cast<size_t>(cols) * 2;
    static bool attr_set[64] = {false};
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    if (dev_id >= 0 && dev_id < 64 && !attr_set[dev_id]) {
      if (cudaFuncSetAttribute(layernorm_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 224 * 1024) !=
          cudaSuccess)
        return record_cuda(cudaGetLastError());
      attr_set[dev_id] = true;
    }
    int* err = device_error_word();
    if (err == nullptr) return record_cuda(cudaErrorInvalidDevice);
    const int64_t want = (rows + nw - 1) / nw;
    const unsigned grid = static_cast<unsigned>(want < num_sms() ? want : num_sms());
    layernorm_fp8_kernel<<<grid, 32 * nw, smem, st>>>(
        static_cast<const __nv_bfloat16*>(x), rows, cols, gamma, beta, eps, fmt == TE_E5M2, scale, q_row,
        static_cast<__nv_bfloat16*>(ln_out), mu, rsigma, amax_out, err);
    count_launch();
    s = launch_status();
    if (s != TE_OK) return s;
  }
  if (scale_inv_out != nullptr) {
    TileArgs a{};   // publishes 1 / scale through the quantizer's own path: an empty launch
    a.scale = scale;
    a.scale_inv_out = scale_inv_out;
    a.fmax = fmt == TE_E4M3 ? 448.0f : 57344.0f;
    s = launch_qtile_any<kQE4M3, false>(x, TE_BF16, 0, cols, nullptr, nullptr, a, st);
  }
  return s;
}

te_status te_quantize_mxfp8(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, uint8_t* q_row,
                            uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, void* stream) {
  te_status s = check_2d(x, in_dtype, rows, cols);
  if (s != TE_OK) return s;
  if ((q_row == nullptr) != (s_row == nullptr) || (q_col == nullptr) != (s_col == nullptr)) return TE_ERR_NULL;
  if ((q_row && cols % 32) || (q_col && rows % 32)) return TE_ERR_SHAPE;
  if ((q_row && (!aligned16(q_row) || !aligned16(s_row))) || (q_col && (!aligned16(q_col) || !aligned16(s_col))))
    return TE_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (q_row && (s = zero_scales(s_row, TE_E8M0, rows, cols, st)) != TE_OK) return s;
  if (q_col && (s = zero_scales(s_col, TE_E8M0, cols, rows, st)) != TE_OK) return s;
  if (rows * cols == 0 || (!q_row && !q_col)) return TE_OK;
  TileArgs a{};
  a.R = rows;
  a.C = cols;
  a.s_row = s_row;
  a.s_col = s_col;
  a.kpad_row = kpad_of(TE_E8M0, cols);
  a.kpad_col = kpad_of(TE_E8M0, rows);
  return launch_qtile_any<kQMX, false>(x, in_dtype, rows, cols, q_row, q_col, a, st);
}

te_status te_quantize_nvfp4(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, uint32_t flags,
                            uint32_t rht_signs, uint64_t seed, uint64_t offset, const float* amax,
                            const float* amax_rht, uint8_t* q_row, uint8_t* s_row, float* gdec_row, uint8_t* q_col,
                            uint8_t* s_col, float* gdec_col, void* stream) {
  te_status s = check_2d(x, in_dtype, rows, cols);
  if (s != TE_OK) return s;
  if (flags & ~7u) return TE_ERR_ARG;
  if ((flags & TE_NVFP4_2D) && (flags & TE_NVFP4_RHT_COL)) return TE_ERR_ARG;
  const bool row = q_row != nullptr, col = q_col != nullptr;
  if (row != (s_row != nullptr) || row != (gdec_row != nullptr)) return TE_ERR_NULL;
  if (col != (s_col != nullptr) || col != (gdec_col != nullptr)) return TE_ERR_NULL;
  if ((row || (col && !(flags & TE_NVFP4_RHT_COL))) && amax == nullptr) return TE_ERR_NULL;
  if (col && (flags & TE_NVFP4_RHT_COL) && amax_rht == nullptr) return TE_ERR_NULL;
  if ((row && cols % 32) || (col && rows % 32)) return TE_ERR_SHAPE;
  if ((row && (!aligned16(q_row) || !aligned16(s_row))) || (col && (!aligned16(q_col) || !aligned16(s_col))))
    return TE_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (row && (s = zero_scales(s_row, TE_UE4M3, rows, cols, st)) != TE_OK) return s;
  if (col && (s = zero_scales(s_col, TE_UE4M3, cols, rows, st)) != TE_OK) return s;
  if (!row && !col) return TE_OK;
  // An empty tensor launches one load-free CTA that publishes the S_dec outputs.
  TileArgs a{};
  a.R = rows;
  a.C = cols;
  a.s_row = s_row;
  a.s_col = s_col;
  a.kpad_row = kpad_of(TE_UE4M3, cols);
  a.kpad_col = kpad_of(TE_UE4M3, rows);
  a.flags = flags;
  a.signs = rht_signs & 0xFFFFu;
  a.seed_lo = static_cast<uint32_t>(seed);
  a.seed_hi = static_cast<uint32_t>(seed >> 32);
  for (int i = 0; i < 10; ++i) {   // the Philox key schedule: bumped by the Weyl constants each round
    a.rk0[i] = a.seed_lo + static_cast<uint32_t>(i) * 0x9E3779B9u;
    a.rk1[i] = a.seed_hi + static_cast<uint32_t>(i) * 0xBB67AE85u;
  }
  a.off_lo = static_cast<uint32_t>(offset);
  a.off_hi = static_cast<uint32_t>(offset >> 32);
  a.amax = amax;
  a.amax_rht = amax_rht;
  a.gdec_row = gdec_row;
  a.gdec_col = gdec_col;
  if (flags & TE_NVFP4_SR) return launch_qtile_any<kQNV, true>(x, in_dtype, rows, cols, q_row, q_col, a, st);
  return launch_qtile_any<kQNV, false>(x, in_dtype, rows, cols, q_row, q_col, a, st);
}

}  // extern "C"

// ---- allocation-free bias-gradient quantization --------------------------------------------------
// Some callers cannot allocate device memory at the point where they quantize dY: code
// that runs while a memory pool is locked or sized up front, or a host runtime that owns
// every allocation and hands the library only the tensors it computes on.  For them the
// workspace of te_quantize_fp8_dbias lives in this fixed array instead (4 MiB, one per
// GPU that loads the library, held until the process exits).
namespace {
constexpr size_t kNoAllocScratchFloats = size_t(1) << 20;
static __device__ __align__(256) float g_dbias_scratch[kNoAllocScratchFloats];

std::mutex g_scratch_mu;
float* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device: host code sees only a
// host-side stand-in for the array's name, so the address is looked up once per device,
// with that device current, and kept.
cudaError_t scratch_address(float** out) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[d] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dbias_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[d] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[d];
  return cudaSuccess;
}
}  // namespace

extern "C" te_status te_quantize_fp8_dbias_noalloc(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols,
                                                   te_dtype fmt, const float* scale, int compute_scale, uint8_t* q_row,
                                                   uint8_t* q_col, float* amax_out, float* scale_inv_out,
                                                   float* dbias, void* stream) {
  // every argument check runs before the scratch address is looked up (that lookup may
  // initialise the device context), so a bad call returns its TE_ERR_* and touches nothing
  te_status s = check_fp8_cast(x, in_dtype, rows, cols, fmt, scale, compute_scale, q_row, q_col, amax_out, dbias);
  if (s != TE_OK) return s;
  if (dbias != nullptr && te_dbias_workspace_bytes(rows, cols) > kNoAllocScratchFloats * sizeof(float))
    return TE_ERR_SHAPE;  // more 64-row-tile partial sums than the fixed scratch holds
  float* ws = nullptr;
  if (dbias != nullptr && rows * cols > 0) {
    const cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess) return record_cuda(e);
  }
  return te_quantize_fp8_dbias(x, in_dtype, rows, cols, fmt, scale, compute_scale, q_row, q_col, amax_out,
                               scale_inv_out, dbias, ws, kNoAllocScratchFloats * sizeof(float), stream);
}
