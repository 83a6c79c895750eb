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

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    if (i) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Stochastic rounding of v to E2M1: the magnitude moves up to the next grid
// point iff r16 * 2^-16 < (|v| - lo) / (hi - lo); |v| >= 6 saturates.
__device__ __forceinline__ uint32_t e2m1_sr(float v, uint32_t r16) {
  const float a = fabsf(v);
  const uint32_t sign = (__float_as_uint(v) >> 31) << 3;
  if (a >= 6.0f) return sign | 7u;
  float lo, inv_span;
  uint32_t code;
  if (a < 0.5f) { lo = 0.0f; inv_span = 2.0f; code = 0; }
  else if (a < 1.0f) { lo = 0.5f; inv_span = 2.0f; code = 1; }
  else if (a < 1.5f) { lo = 1.0f; inv_span = 2.0f; code = 2; }
  else if (a < 2.0f) { lo = 1.5f; inv_span = 2.0f; code = 3; }
  else if (a < 3.0f) { lo = 2.0f; inv_span = 1.0f; code = 4; }
  else if (a < 4.0f) { lo = 3.0f; inv_span = 1.0f; code = 5; }
  else { lo = 4.0f; inv_span = 0.5f; code = 6; }
  const float frac = __fmul_rn(__fsub_rn(a, lo), inv_span);  // exact
  const float thr = __fmul_rn(static_cast<float>(r16), 1.52587890625e-5f);  // exact: r16 * 2^-16
  return sign | (thr < frac ? code + 1u : code);
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
template <>
struct Chunk<__nv_bfloat16, 8> {
  using Raw = uint2;
  static constexpr int N = 4;
};
template <>
struct Chunk<float, 8> {
  using Raw = uint2;
  static constexpr int N = 2;
};

__device__ __forceinline__ uint4 ld_raw(const uint4* p) { return __ldg(p); }
__device__ __forceinline__ uint2 ld_raw(const uint2* p) { return __ldg(p); }
__device__ __forceinline__ void zero_raw(uint4& r) { r = make_uint4(0, 0, 0, 0); }
__device__ __forceinline__ void zero_raw(uint2& r) { r = make_uint2(0, 0); }
__device__ __forceinline__ uint32_t raw_word(const uint4& r, int k) {
  return k == 0 ? r.x : (k == 1 ? r.y : (k == 2 ? r.z : r.w));
}
__device__ __forceinline__ uint32_t raw_word(const uint2& r, int k) { return k == 0 ? r.x : r.y; }

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
  Patch<T, 16, 16> p;
  p.load(x, R, C);
  block_max_to(p.absmax(), amax);
  if (RHT) {
    float mr = 0.0f;
#pragma unroll
    for (int i = 0; i < Patch<T, 16, 16>::PC; ++i) {
      float col[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) col[r] = p.at(r, i);
      rht16(col, signs);
#pragma unroll
      for (int r = 0; r < 16; ++r) mr = fmaxf(mr, fabsf(col[r]));
    }
    block_max_to(mr, amax_rht);
  }
}

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
    eff = h[0];
    for (int j = 1; j < L; ++j) eff = fmaxf(eff, h[j]);
  }
  float s = scale[i];
  if (isfinite(eff) && eff > 0.0f) {
    const float t = __fmul_rn(__fdiv_rn(fmax, eff), margin_mul);
    if (isfinite(t)) s = t;
  }
  scale[i] = s;
  scale_inv[i] = __fdiv_rn(1.0f, s);
}

__device__ __forceinline__ float current_scale(float a, float fmax) {
  if (!(isfinite(a) && a > 0.0f)) return 1.0f;
  const float s = __fdiv_rn(fmax, a);
  return isfinite(s) ? s : 1.0f;
}

// ---- FP8 ----------------------------------------------------------------------------------------
struct Fp8Args {
  int64_t R, C;
  const float* scale;     // Delayed: the scale to use
  const float* amax_in;   // Current: the tensor amax
  int current;
  float fmax;
  uint8_t* q_row;
  uint8_t* q_col;
  float* amax_out;        // Delayed: fused amax (nullable)
  float* scale_inv_out;   // nullable
};

template <bool E5M2>
__device__ __forceinline__ uint32_t fp8x2(float a, float b) {
  return E5M2 ? cvt_e5m2x2(a, b) : cvt_e4m3x2(a, b);
}

template <typename T, bool E5M2>
__global__ void __launch_bounds__(kThreads, 2) fp8_kernel(const T* __restrict__ x, Fp8Args a) {
  using P = Patch<T, 16, 16>;
  constexpr int PC = P::PC;
  P p;
  p.load(x, a.R, a.C);
  const float s = a.current ? current_scale(*a.amax_in, a.fmax) : *a.scale;
  if (p.live && a.q_row != nullptr) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      uint32_t w[PC / 4];
#pragma unroll
      for (int j = 0; j < PC / 4; ++j) {
        const uint32_t lo = fp8x2<E5M2>(__fmul_rn(p.at(r, 4 * j), s), __fmul_rn(p.at(r, 4 * j + 1), s));
        const uint32_t hi = fp8x2<E5M2>(__fmul_rn(p.at(r, 4 * j + 2), s), __fmul_rn(p.at(r, 4 * j + 3), s));
        w[j] = lo | (hi << 16);
      }
      uint8_t* dst = a.q_row + (p.r0 + r) * a.C + p.c0;
      if (PC == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[PC / 4 - 1]);
      else *reinterpret_cast<uint32_t*>(dst) = w[0];
    }
  }
  if (p.live && a.q_col != nullptr) {
#pragma unroll
    for (int i = 0; i < PC; ++i) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = fp8x2<E5M2>(__fmul_rn(p.at(4 * j, i), s), __fmul_rn(p.at(4 * j + 1, i), s));
        const uint32_t hi = fp8x2<E5M2>(__fmul_rn(p.at(4 * j + 2, i), s), __fmul_rn(p.at(4 * j + 3, i), s));
        w[j] = lo | (hi << 16);
      }
      *reinterpret_cast<uint4*>(a.q_col + (p.c0 + i) * a.R + p.r0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  if (a.scale_inv_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *a.scale_inv_out = __fdiv_rn(1.0f, s);
  if (a.amax_out != nullptr) block_max_to(p.absmax(), a.amax_out);
}

// ---- MXFP8 ----------------------------------------------------------------------------------------
// Shared exponent of a block: clamp(floor(log2 amax) - 8, -127, 127); -127 for a zero block.
__device__ __forceinline__ int mx_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  if (b == 0) return -127;
  const uint32_t ef = b >> 23;
  int e = (ef == 0) ? (31 - __clz(static_cast<int>(b))) - 149 : static_cast<int>(ef) - 127;
  e -= 8;
  return max(-127, min(127, e));
}
__device__ __forceinline__ float mx_mult(int E) { return __uint_as_float(static_cast<uint32_t>(127 - E) << 23); }

struct MxArgs {
  int64_t R, C;
  uint8_t* q_row;
  uint8_t* s_row;
  int64_t kpad_row;  // padded scale columns of the row copy
  uint8_t* q_col;
  uint8_t* s_col;
  int64_t kpad_col;
};

// PR = 32 when the col copy is requested (one column block per patch), else 16.
template <typename T, int PR>
__global__ void __launch_bounds__(kThreads, 2) mxfp8_kernel(const T* __restrict__ x, MxArgs a) {
  using P = Patch<T, 8, PR>;
  constexpr int PC = P::PC;
  constexpr int LANES = 32 / PC;  // threads sharing one row block of 32
  P p;
  p.load(x, a.R, a.C);
  if (a.q_row != nullptr) {
    const bool first = ((p.c0 / PC) % LANES) == 0;
#pragma unroll
    for (int r = 0; r < PR; ++r) {
      float m = 0.0f;
#pragma unroll
      for (int i = 0; i < PC; ++i) m = fmaxf(m, fabsf(p.at(r, i)));
      m = group_max<LANES>(m);
      const int E = mx_exponent(m);
      const float mult = mx_mult(E);
      uint32_t w = 0;
#pragma unroll
      for (int j = 0; j < PC / 2; ++j)
        w |= cvt_e4m3x2(__fmul_rn(p.at(r, 2 * j), mult), __fmul_rn(p.at(r, 2 * j + 1), mult)) << (16 * j);
      if (p.live) {
        uint8_t* dst = a.q_row + (p.r0 + r) * a.C + p.c0;
        if (PC == 4) *reinterpret_cast<uint32_t*>(dst) = w;
        else *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(w);
        if (first) a.s_row[scale_offset(p.r0 + r, p.c0 / 32, a.kpad_row)] = static_cast<uint8_t>(E + 127);
      }
    }
  }
  if (PR == 32 && a.q_col != nullptr && p.live) {
#pragma unroll
    for (int i = 0; i < PC; ++i) {
      float m = 0.0f;
#pragma unroll
      for (int r = 0; r < PR; ++r) m = fmaxf(m, fabsf(p.at(r, i)));
      const int E = mx_exponent(m);
      const float mult = mx_mult(E);
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(p.at(4 * j, i), mult), __fmul_rn(p.at(4 * j + 1, i), mult));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(p.at(4 * j + 2, i), mult), __fmul_rn(p.at(4 * j + 3, i), mult));
        w[j] = lo | (hi << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(a.q_col + (p.c0 + i) * a.R + p.r0);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      a.s_col[scale_offset(p.c0 + i, p.r0 / 32, a.kpad_col)] = static_cast<uint8_t>(E + 127);
    }
  }
}

// ---- NVFP4 ----------------------------------------------------------------------------------------
struct NvArgs {
  int64_t R, C;
  uint32_t flags, signs;
  uint32_t seed_lo, seed_hi, off_lo, off_hi;
  const float* amax;
  const float* amax_rht;
  uint8_t* q_row;
  uint8_t* s_row;
  float* gdec_row;
  int64_t kpad_row;
  uint8_t* q_col;
  uint8_t* s_col;
  float* gdec_col;
  int64_t kpad_col;
};

__device__ __forceinline__ float nv_senc(float A) {
  if (!(A > 0.0f)) return 1.0f;
  const float s = __fdiv_rn(2688.0f, A);
  return isfinite(s) ? s : 1.0f;
}

// UE4M3 block-scale code of a block with amax bm: RN(fl32(fl32(bm / 6) * S_enc)).
__device__ __forceinline__ uint32_t nv_scale_code(float bm, float senc) {
  return cvt_e4m3x2(__fmul_rn(__fdiv_rn(bm, 6.0f), senc), 0.0f) & 0x7Fu;
}

// The 16-bit random values of the 8 elements g8*8 .. g8*8+7 of a copy (element
// 2k + h takes half h of word k of Philox(counter = (g8, copy, offset))).
__device__ __forceinline__ uint4 nv_rand8(const NvArgs& a, uint64_t g8, uint32_t copy_id) {
  return philox4x32_10(make_uint4(static_cast<uint32_t>(g8), copy_id, a.off_lo, a.off_hi), a.seed_lo, a.seed_hi);
}
__device__ __forceinline__ uint32_t rand16_of(const uint4& w, int k) {  // k = element index within the 8
  const uint32_t word = raw_word(w, k >> 1);
  return (k & 1) ? (word >> 16) : (word & 0xFFFFu);
}

template <typename T, bool SR>
__global__ void __launch_bounds__(kThreads, 2) nvfp4_kernel(const T* __restrict__ x, NvArgs a) {
  using P = Patch<T, 16, 16>;
  constexpr int PC = P::PC;
  constexpr int LANES = 16 / PC;  // threads sharing one row block of 16
  __shared__ float rtab[2][128];  // r = fl32(S_enc / dec(code)) for the row / col copy
  const bool do_row = a.q_row != nullptr, do_col = a.q_col != nullptr;
  const bool two_d = (a.flags & TE_NVFP4_2D) != 0, rht = (a.flags & TE_NVFP4_RHT_COL) != 0;
  const float senc_r = do_row ? nv_senc(*a.amax) : 1.0f;
  const float senc_c = do_col ? nv_senc(rht ? *a.amax_rht : *a.amax) : 1.0f;
  if (threadIdx.x < 128) {
    const float dv = ue4m3_value(threadIdx.x);
    rtab[0][threadIdx.x] = dv > 0.0f ? __fdiv_rn(senc_r, dv) : 0.0f;
    rtab[1][threadIdx.x] = dv > 0.0f ? __fdiv_rn(senc_c, dv) : 0.0f;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (do_row && a.gdec_row != nullptr) *a.gdec_row = __fdiv_rn(1.0f, senc_r);
    if (do_col && a.gdec_col != nullptr) *a.gdec_col = __fdiv_rn(1.0f, senc_c);
  }
  P p;
  p.load(x, a.R, a.C);
  __syncthreads();
  float tile_max = 0.0f;  // 2D: amax of the 16 x 16 tile this patch belongs to
  if (two_d) tile_max = group_max<LANES>(p.absmax());

  if (do_row) {
    const bool first = ((p.c0 / PC) % LANES) == 0;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float m = 0.0f;
      if (!two_d) {
#pragma unroll
        for (int i = 0; i < PC; ++i) m = fmaxf(m, fabsf(p.at(r, i)));
        m = group_max<LANES>(m);
      } else {
        m = tile_max;
      }
      const uint32_t sc = nv_scale_code(m, senc_r);
      const float rr = rtab[0][sc];
      const uint64_t g = static_cast<uint64_t>(p.r0 + r) * static_cast<uint64_t>(a.C) + static_cast<uint64_t>(p.c0);
      uint32_t w = 0;
      if (!SR) {
#pragma unroll
        for (int j = 0; j < PC / 2; ++j)
          w |= cvt_e2m1x2(__fmul_rn(p.at(r, 2 * j), rr), __fmul_rn(p.at(r, 2 * j + 1), rr)) << (8 * j);
      } else {
        const uint4 rnd = nv_rand8(a, g >> 3, 0u);
        const int k0 = static_cast<int>(g & 7);
#pragma unroll
        for (int i = 0; i < PC; ++i) w |= e2m1_sr(__fmul_rn(p.at(r, i), rr), rand16_of(rnd, k0 + i)) << (4 * i);
      }
      if (p.live) {
        uint8_t* dst = a.q_row + (p.r0 + r) * (a.C / 2) + p.c0 / 2;
        if (PC == 8) *reinterpret_cast<uint32_t*>(dst) = w;
        else *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(w);
        if (first) a.s_row[scale_offset(p.r0 + r, p.c0 / 16, a.kpad_row)] = static_cast<uint8_t>(sc);
      }
    }
  }
  if (do_col && p.live) {
#pragma unroll
    for (int i = 0; i < PC; ++i) {
      float v[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) v[r] = p.at(r, i);
      if (rht) rht16(v, a.signs);
      float m = tile_max;
      if (!two_d) {
        m = 0.0f;
#pragma unroll
        for (int r = 0; r < 16; ++r) m = fmaxf(m, fabsf(v[r]));
      }
      const uint32_t sc = nv_scale_code(m, senc_c);
      const float rr = rtab[1][sc];
      uint32_t lo = 0, hi = 0;
      if (!SR) {
#pragma unroll
        for (int j = 0; j < 4; ++j) lo |= cvt_e2m1x2(__fmul_rn(v[2 * j], rr), __fmul_rn(v[2 * j + 1], rr)) << (8 * j);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          hi |= cvt_e2m1x2(__fmul_rn(v[8 + 2 * j], rr), __fmul_rn(v[8 + 2 * j + 1], rr)) << (8 * j);
      } else {
        const uint64_t g = static_cast<uint64_t>(p.c0 + i) * static_cast<uint64_t>(a.R) + static_cast<uint64_t>(p.r0);
        const uint4 r0 = nv_rand8(a, g >> 3, 1u);
        const uint4 r1 = nv_rand8(a, (g >> 3) + 1, 1u);
#pragma unroll
        for (int k = 0; k < 8; ++k) lo |= e2m1_sr(__fmul_rn(v[k], rr), rand16_of(r0, k)) << (4 * k);
#pragma unroll
        for (int k = 0; k < 8; ++k) hi |= e2m1_sr(__fmul_rn(v[8 + k], rr), rand16_of(r1, k)) << (4 * k);
      }
      *reinterpret_cast<uint2*>(a.q_col + (p.c0 + i) * (a.R / 2) + p.r0 / 2) = make_uint2(lo, hi);
      a.s_col[scale_offset(p.c0 + i, p.r0 / 16, a.kpad_col)] = static_cast<uint8_t>(sc);
    }
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
  if (cudaMemsetAsync(amax, 0, sizeof(float), st) != cudaSuccess) return record_cuda(cudaGetLastError());
  if (amax_rht != nullptr && cudaMemsetAsync(amax_rht, 0, sizeof(float), st) != cudaSuccess)
    return record_cuda(cudaGetLastError());
  if (rows * cols == 0) return TE_OK;
  if (in == TE_BF16) {
    const auto* p = static_cast<const __nv_bfloat16*>(x);
    const unsigned blocks = patch_blocks(rows, cols, 16, 8);
    if (amax_rht) amax_kernel<__nv_bfloat16, true><<<blocks, kThreads, 0, st>>>(p, rows, cols, amax, amax_rht, signs);
    else amax_kernel<__nv_bfloat16, false><<<blocks, kThreads, 0, st>>>(p, rows, cols, amax, nullptr, signs);
  } else {
    const auto* p = static_cast<const float*>(x);
    const unsigned blocks = patch_blocks(rows, cols, 16, 4);
    if (amax_rht) amax_kernel<float, true><<<blocks, kThreads, 0, st>>>(p, rows, cols, amax, amax_rht, signs);
    else amax_kernel<float, false><<<blocks, kThreads, 0, st>>>(p, rows, cols, amax, nullptr, signs);
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

inline int vec_elems(te_dtype in, int bytes) { return bytes / (in == TE_BF16 ? 2 : 4); }

}  // namespace
}  // namespace te

using namespace te;

extern "C" {

te_status te_amax_reduce(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, float* amax, float* amax_rht,
                         uint32_t rht_signs, void* stream) {
  te_status s = check_2d(x, in_dtype, rows, cols);
  if (s != TE_OK) return s;
  if (amax == nullptr) return TE_ERR_NULL;
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

te_status te_quantize_fp8(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, te_dtype fmt,
                          const float* scale, int compute_scale, uint8_t* q_row, uint8_t* q_col, float* amax_out,
                          float* scale_inv_out, void* stream) {
  te_status s = check_2d(x, in_dtype, rows, cols);
  if (s != TE_OK) return s;
  if (fmt != TE_E4M3 && fmt != TE_E5M2) return TE_ERR_DTYPE;
  if (compute_scale != 0 && compute_scale != 1) return TE_ERR_ARG;
  if (compute_scale ? amax_out == nullptr : scale == nullptr) return TE_ERR_NULL;
  if ((q_row && !aligned16(q_row)) || (q_col && !aligned16(q_col))) return TE_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (compute_scale) {
    s = launch_amax(x, in_dtype, rows, cols, amax_out, nullptr, 0, st);
    if (s != TE_OK) return s;
  } else if (amax_out != nullptr) {
    if (cudaMemsetAsync(amax_out, 0, sizeof(float), st) != cudaSuccess) return record_cuda(cudaGetLastError());
  }
  if (rows * cols == 0 && scale_inv_out == nullptr) return TE_OK;
  // An empty tensor still launches one (load-free) block so that scale_inv_out is published.
  Fp8Args a{rows, cols, scale, amax_out, compute_scale, fmt == TE_E4M3 ? 448.0f : 57344.0f, q_row, q_col,
            compute_scale ? nullptr : amax_out, scale_inv_out};
  const unsigned blocks = patch_blocks(rows, cols, 16, vec_elems(in_dtype, 16));
  if (in_dtype == TE_BF16) {
    const auto* p = static_cast<const __nv_bfloat16*>(x);
    if (fmt == TE_E4M3) fp8_kernel<__nv_bfloat16, false><<<blocks, kThreads, 0, st>>>(p, a);
    else fp8_kernel<__nv_bfloat16, true><<<blocks, kThreads, 0, st>>>(p, a);
  } else {
    const auto* p = static_cast<const float*>(x);
    if (fmt == TE_E4M3) fp8_kernel<float, false><<<blocks, kThreads, 0, st>>>(p, a);
    else fp8_kernel<float, true><<<blocks, kThreads, 0, st>>>(p, a);
  }
  count_launch();
  return launch_status();
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
  MxArgs a{rows, cols, q_row, s_row, kpad_of(TE_E8M0, cols), q_col, s_col, kpad_of(TE_E8M0, rows)};
  const int pc = vec_elems(in_dtype, 8);
  if (q_col) {
    const unsigned blocks = patch_blocks(rows, cols, 32, pc);
    if (in_dtype == TE_BF16) mxfp8_kernel<__nv_bfloat16, 32><<<blocks, kThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(x), a);
    else mxfp8_kernel<float, 32><<<blocks, kThreads, 0, st>>>(static_cast<const float*>(x), a);
  } else {
    const unsigned blocks = patch_blocks(rows, cols, 16, pc);
    if (in_dtype == TE_BF16) mxfp8_kernel<__nv_bfloat16, 16><<<blocks, kThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(x), a);
    else mxfp8_kernel<float, 16><<<blocks, kThreads, 0, st>>>(static_cast<const float*>(x), a);
  }
  count_launch();
  return launch_status();
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
  if ((row && (!aligned16(q_row) || !aligned16(s_row))) || (col && (!aligned16(q_col) || !aligned16(s_col))))
    return TE_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (row && (s = zero_scales(s_row, TE_UE4M3, rows, cols, st)) != TE_OK) return s;
  if (col && (s = zero_scales(s_col, TE_UE4M3, cols, rows, st)) != TE_OK) return s;
  if (!row && !col) return TE_OK;
  // An empty tensor launches one load-free block that publishes the S_dec outputs.
  NvArgs a{rows, cols, flags, rht_signs & 0xFFFFu,
           static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32),
           static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32),
           amax, amax_rht, q_row, s_row, gdec_row, kpad_of(TE_UE4M3, cols),
           q_col, s_col, gdec_col, kpad_of(TE_UE4M3, rows)};
  const bool sr = (flags & TE_NVFP4_SR) != 0;
  const unsigned blocks = patch_blocks(rows, cols, 16, vec_elems(in_dtype, 16));
  if (in_dtype == TE_BF16) {
    const auto* p = static_cast<const __nv_bfloat16*>(x);
    if (sr) nvfp4_kernel<__nv_bfloat16, true><<<blocks, kThreads, 0, st>>>(p, a);
    else nvfp4_kernel<__nv_bfloat16, false><<<blocks, kThreads, 0, st>>>(p, a);
  } else {
    const auto* p = static_cast<const float*>(x);
    if (sr) nvfp4_kernel<float, true><<<blocks, kThreads, 0, st>>>(p, a);
    else nvfp4_kernel<float, false><<<blocks, kThreads, 0, st>>>(p, a);
  }
  count_launch();
  return launch_status();
}

}  // extern "C"
