// Quantizer kernels: per-tensor amax (plain and after the 16-point random
// Hadamard transform), the DelayedScaling history/scale update, and the FP8,
// MXFP8 and NVFP4 quantizers that write the row-wise and column-wise
// (transposed) copies of a tensor from a single read.
//
// Every quantizer works on 64 x 64 tiles staged once in shared memory as fp32:
// the row copy is produced from tile rows, the col copy from tile columns, so
// the input is read from HBM exactly once.  Loads are 16-byte vectors, coalesced
// along the row; stores of both copies are 16-byte (FP8/MXFP8) or 8-byte (NVFP4)
// vectors.  All code-deciding arithmetic is IEEE fp32 round-to-nearest-even
// (compiled with -fmad=false) so the codes are bit-identical to the definitions
// in te_gb300.h.
#include <cuda_bf16.h>
#include <string.h>

#include "common.cuh"

namespace te {
namespace {

constexpr int kTile = 64;
constexpr int kThreads = 256;

// ---- element access ----------------------------------------------------------------

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

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
// point iff (w >> 8) * 2^-24 < (|v| - lo) / (hi - lo); |v| >= 6 saturates.
__device__ __forceinline__ uint32_t e2m1_sr(float v, uint32_t w) {
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
  const float thr = __fmul_rn(static_cast<float>(w >> 8), 5.9604644775390625e-8f);  // exact: k * 2^-24
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
}

// ---- amax ---------------------------------------------------------------------------------------
// Each thread reads a 16-row x 8-column patch (sixteen coalesced 16-byte loads),
// takes the plain amax and, with RHT, the amax of the 8 transformed columns.
template <typename T, bool RHT>
__global__ void __launch_bounds__(kThreads) amax_kernel(const T* __restrict__ x, int64_t R, int64_t C, float* amax,
                                                        float* amax_rht, uint32_t signs) {
  const int64_t ncg = C / 8;
  const int64_t total = (R / 16) * ncg;
  float m = 0.0f, mr = 0.0f;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t band = idx / ncg, cg = idx - band * ncg;
    const T* p = x + band * 16 * C + cg * 8;
    float v[16][8];
#pragma unroll
    for (int r = 0; r < 16; ++r) load8(p + r * C, v[r]);
#pragma unroll
    for (int r = 0; r < 16; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) m = fmaxf(m, fabsf(v[r][c]));
    if (RHT) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float col[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) col[r] = v[r][c];
        rht16(col, signs);
#pragma unroll
        for (int r = 0; r < 16; ++r) mr = fmaxf(mr, fabsf(col[r]));
      }
    }
  }
  block_max_to(m, amax);
  if (RHT) {
    __syncthreads();
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

// ---- tile staging ---------------------------------------------------------------------------------
// Loads the 64 x 64 tile at (r0, c0) into smem as fp32 (zeros outside [R, C]) and
// returns the thread's partial amax.  Thread t loads rows t/8 and t/8 + 32,
// columns (t % 8) * 8 .. + 7.
template <typename T>
__device__ __forceinline__ float stage_tile(const T* __restrict__ x, int64_t R, int64_t C, int64_t r0, int64_t c0,
                                            float (*tile)[kTile + 1]) {
  const int t = threadIdx.x;
  const int cc = (t & 7) * 8;
  float m = 0.0f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int rr = (t >> 3) + 32 * h;
    const int64_t r = r0 + rr, c = c0 + cc;
    float v[8];
    if (r < R && c < C) {
      load8(x + r * C + c, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      tile[rr][cc + i] = v[i];
      m = fmaxf(m, fabsf(v[i]));
    }
  }
  return m;
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

template <typename T, bool E5M2>
__global__ void __launch_bounds__(kThreads) fp8_kernel(const T* __restrict__ x, Fp8Args a) {
  __shared__ float tile[kTile][kTile + 1];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTile, c0 = static_cast<int64_t>(blockIdx.x) * kTile;
  const float lmax = stage_tile(x, a.R, a.C, r0, c0, tile);
  const float s = a.current ? current_scale(*a.amax_in, a.fmax) : *a.scale;
  __syncthreads();
  const int t = threadIdx.x;
  const int lane_row = t >> 2, seg = (t & 3) * 16;
  if (a.q_row != nullptr) {
    const int64_t r = r0 + lane_row, c = c0 + seg;
    if (r < a.R && c < a.C) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = tile[lane_row][seg + i];
      *reinterpret_cast<uint4*>(a.q_row + r * a.C + c) = pack_fp8_16<E5M2>(v, s);
    }
  }
  if (a.q_col != nullptr) {
    const int64_t c = c0 + lane_row, r = r0 + seg;
    if (c < a.C && r < a.R) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = tile[seg + i][lane_row];
      *reinterpret_cast<uint4*>(a.q_col + c * a.R + r) = pack_fp8_16<E5M2>(v, s);
    }
  }
  if (a.scale_inv_out != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && t == 0)
    *a.scale_inv_out = __fdiv_rn(1.0f, s);
  if (a.amax_out != nullptr) block_max_to(lmax, a.amax_out);
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

struct MxArgs {
  int64_t R, C;
  uint8_t* q_row;
  uint8_t* s_row;
  int64_t kpad_row;  // padded scale columns of the row copy
  uint8_t* q_col;
  uint8_t* s_col;
  int64_t kpad_col;
};

// One block of 32 is handled by two threads (16 elements each) that are lanes
// t and t^1; it writes the codes and returns the scale byte.
__device__ __forceinline__ uint32_t mx_quantize_half(const float (&v)[16], uint4* dst, bool valid) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  const int E = mx_exponent(m);
  const float mult = __uint_as_float(static_cast<uint32_t>(127 - E) << 23);
  if (valid) *dst = pack_fp8_16<false>(v, mult);
  return static_cast<uint32_t>(E + 127);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) mxfp8_kernel(const T* __restrict__ x, MxArgs a) {
  __shared__ float tile[kTile][kTile + 1];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTile, c0 = static_cast<int64_t>(blockIdx.x) * kTile;
  stage_tile(x, a.R, a.C, r0, c0, tile);
  __syncthreads();
  const int t = threadIdx.x;
  const int lane_row = t >> 2, sub = t & 3, seg = sub * 16;
  if (a.q_row != nullptr) {
    const int64_t r = r0 + lane_row, c = c0 + seg;
    const bool valid = r < a.R && c < a.C;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = tile[lane_row][seg + i];
    const uint32_t sb = mx_quantize_half(v, reinterpret_cast<uint4*>(a.q_row + r * a.C + c), valid);
    const uint32_t sb_next = __shfl_down_sync(0xFFFFFFFFu, sb, 2);  // block of columns 32..63
    if (sub == 0 && r < a.R) {
      const uint64_t j0 = static_cast<uint64_t>(c0 / 32);
      const uint32_t hi = (c0 + 32 < a.C) ? sb_next : 0u;
      *reinterpret_cast<uint16_t*>(a.s_row + scale_offset(r, j0, a.kpad_row)) = static_cast<uint16_t>(sb | (hi << 8));
    }
  }
  if (a.q_col != nullptr) {
    const int64_t c = c0 + lane_row, r = r0 + seg;
    const bool valid = c < a.C && r < a.R;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = tile[seg + i][lane_row];
    const uint32_t sb = mx_quantize_half(v, reinterpret_cast<uint4*>(a.q_col + c * a.R + r), valid);
    const uint32_t sb_next = __shfl_down_sync(0xFFFFFFFFu, sb, 2);
    if (sub == 0 && c < a.C) {
      const uint64_t j0 = static_cast<uint64_t>(r0 / 32);
      const uint32_t hi = (r0 + 32 < a.R) ? sb_next : 0u;
      *reinterpret_cast<uint16_t*>(a.s_col + scale_offset(c, j0, a.kpad_col)) = static_cast<uint16_t>(sb | (hi << 8));
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

// Quantizes one 16-element block: returns the UE4M3 scale code, writes 8 packed bytes.
// `g0` is the row-major index of v[0] inside the copy (for stochastic rounding).
__device__ __forceinline__ uint32_t nv_quantize_block(const float (&v)[16], float blk_amax, float senc, bool sr,
                                                      const NvArgs& a, uint32_t copy_id, uint64_t g0, uint2* dst,
                                                      bool valid) {
  const float pre = __fmul_rn(__fdiv_rn(blk_amax, 6.0f), senc);
  const uint32_t sc = cvt_e4m3x2(pre, 0.0f) & 0x7Fu;
  const float sv = ue4m3_value(sc);
  const float r = sv > 0.0f ? __fdiv_rn(senc, sv) : 0.0f;
  float y[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(v[i], r);
  uint32_t lo = 0, hi = 0;
  if (!sr) {
#pragma unroll
    for (int i = 0; i < 4; ++i) lo |= cvt_e2m1x2(y[2 * i], y[2 * i + 1]) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) hi |= cvt_e2m1x2(y[8 + 2 * i], y[8 + 2 * i + 1]) << (8 * i);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint64_t grp = (g0 >> 2) + q;
      const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(grp), copy_id, a.off_lo, a.off_hi), a.seed_lo,
                                    a.seed_hi);
      const uint32_t n0 = e2m1_sr(y[4 * q], w.x), n1 = e2m1_sr(y[4 * q + 1], w.y);
      const uint32_t n2 = e2m1_sr(y[4 * q + 2], w.z), n3 = e2m1_sr(y[4 * q + 3], w.w);
      const uint32_t word16 = n0 | (n1 << 4) | (n2 << 8) | (n3 << 12);
      if (q < 2) lo |= word16 << (16 * q);
      else hi |= word16 << (16 * (q - 2));
    }
  }
  if (valid) *dst = make_uint2(lo, hi);
  return sc;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) nvfp4_kernel(const T* __restrict__ x, NvArgs a) {
  __shared__ float tile[kTile][kTile + 1];
  __shared__ float amax2d[4][4];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTile, c0 = static_cast<int64_t>(blockIdx.x) * kTile;
  stage_tile(x, a.R, a.C, r0, c0, tile);
  __syncthreads();
  const int t = threadIdx.x;
  const bool two_d = (a.flags & TE_NVFP4_2D) != 0;
  const bool sr = (a.flags & TE_NVFP4_SR) != 0;
  if (two_d) {
    const int st = t >> 4, sr_ = st >> 2, sc_ = st & 3, rr = t & 15;
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(tile[sr_ * 16 + rr][sc_ * 16 + i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (rr == 0) amax2d[sr_][sc_] = m;
    __syncthreads();
  }
  const int lane_row = t >> 2, sub = t & 3, seg = sub * 16;
  if (a.q_row != nullptr) {
    const float senc = nv_senc(*a.amax);
    const int64_t r = r0 + lane_row, c = c0 + seg;
    const bool valid = r < a.R && c < a.C;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = tile[lane_row][seg + i];
    float bm = 0.0f;
    if (two_d) {
      bm = amax2d[lane_row >> 4][sub];
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) bm = fmaxf(bm, fabsf(v[i]));
    }
    const uint64_t g0 = static_cast<uint64_t>(r) * static_cast<uint64_t>(a.C) + static_cast<uint64_t>(c);
    const uint32_t sc = nv_quantize_block(v, bm, senc, sr, a, 0u, g0,
                                          reinterpret_cast<uint2*>(a.q_row + r * (a.C / 2) + c / 2), valid);
    uint32_t word = sc;
    word |= __shfl_down_sync(0xFFFFFFFFu, sc, 1) << 8;
    word |= __shfl_down_sync(0xFFFFFFFFu, sc, 2) << 16;
    word |= __shfl_down_sync(0xFFFFFFFFu, sc, 3) << 24;
    if (sub == 0 && r < a.R)
      *reinterpret_cast<uint32_t*>(a.s_row + scale_offset(r, static_cast<uint64_t>(c0 / 16), a.kpad_row)) = word;
    if (a.gdec_row != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && t == 0) *a.gdec_row = __fdiv_rn(1.0f, senc);
  }
  if (a.q_col != nullptr) {
    const bool rht = (a.flags & TE_NVFP4_RHT_COL) != 0;
    const float senc = nv_senc(rht ? *a.amax_rht : *a.amax);
    const int64_t c = c0 + lane_row, r = r0 + seg;
    const bool valid = c < a.C && r < a.R;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = tile[seg + i][lane_row];
    if (rht) rht16(v, a.signs);
    float bm = 0.0f;
    if (two_d) {
      bm = amax2d[sub][lane_row >> 4];
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) bm = fmaxf(bm, fabsf(v[i]));
    }
    const uint64_t g0 = static_cast<uint64_t>(c) * static_cast<uint64_t>(a.R) + static_cast<uint64_t>(r);
    const uint32_t sc = nv_quantize_block(v, bm, senc, sr, a, 1u, g0,
                                          reinterpret_cast<uint2*>(a.q_col + c * (a.R / 2) + r / 2), valid);
    uint32_t word = sc;
    word |= __shfl_down_sync(0xFFFFFFFFu, sc, 1) << 8;
    word |= __shfl_down_sync(0xFFFFFFFFu, sc, 2) << 16;
    word |= __shfl_down_sync(0xFFFFFFFFu, sc, 3) << 24;
    if (sub == 0 && c < a.C)
      *reinterpret_cast<uint32_t*>(a.s_col + scale_offset(c, static_cast<uint64_t>(r0 / 16), a.kpad_col)) = word;
    if (a.gdec_col != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && t == 0) *a.gdec_col = __fdiv_rn(1.0f, senc);
  }
}

// ---- host helpers ----------------------------------------------------------------------------------

inline bool in_dtype_ok(te_dtype d) { return d == TE_BF16 || d == TE_F32; }

inline te_status check_2d(const void* x, te_dtype in, int64_t rows, int64_t cols) {
  if (!in_dtype_ok(in)) return TE_ERR_DTYPE;
  if (rows < 0 || cols < 0 || rows % 16 || cols % 16) return TE_ERR_SHAPE;
  if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31)) return TE_ERR_SHAPE;
  if (rows * cols > 0) {
    if (x == nullptr) return TE_ERR_NULL;
    if (!aligned16(x)) return TE_ERR_ALIGN;
  }
  return TE_OK;
}

inline dim3 tile_grid(int64_t rows, int64_t cols) {
  return dim3(static_cast<unsigned>((cols + kTile - 1) / kTile), static_cast<unsigned>((rows + kTile - 1) / kTile));
}

inline bool grid_ok(int64_t rows) { return (rows + kTile - 1) / kTile <= 65535; }

te_status launch_amax(const void* x, te_dtype in, int64_t rows, int64_t cols, float* amax, float* amax_rht,
                      uint32_t signs, cudaStream_t st) {
  if (cudaMemsetAsync(amax, 0, sizeof(float), st) != cudaSuccess) return record_cuda(cudaGetLastError());
  if (amax_rht != nullptr && cudaMemsetAsync(amax_rht, 0, sizeof(float), st) != cudaSuccess)
    return record_cuda(cudaGetLastError());
  if (rows * cols == 0) return TE_OK;
  const int64_t items = (rows / 16) * (cols / 8);
  const int64_t want = (items + kThreads - 1) / kThreads;
  const unsigned blocks = static_cast<unsigned>(want < 1 ? 1 : (want > 65535 * 8 ? 65535 * 8 : want));
  if (in == TE_BF16) {
    const auto* p = static_cast<const __nv_bfloat16*>(x);
    if (amax_rht) amax_kernel<__nv_bfloat16, true><<<blocks, kThreads, 0, st>>>(p, rows, cols, amax, amax_rht, signs);
    else amax_kernel<__nv_bfloat16, false><<<blocks, kThreads, 0, st>>>(p, rows, cols, amax, nullptr, signs);
  } else {
    const auto* p = static_cast<const float*>(x);
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

}  // namespace
}  // namespace te

using namespace te;

extern "C" {

te_status te_amax_reduce(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, float* amax, float* amax_rht,
                         uint32_t rht_signs, void* stream) {
  te_status s = check_2d(x, in_dtype, rows, cols);
  if (s != TE_OK) return s;
  if (amax == nullptr) return TE_ERR_NULL;
  return launch_amax(x, in_dtype, rows, cols, amax, amax_rht, rht_signs, static_cast<cudaStream_t>(stream));
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
  if (!grid_ok(rows)) return TE_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (compute_scale) {
    s = launch_amax(x, in_dtype, rows, cols, amax_out, nullptr, 0, st);
    if (s != TE_OK) return s;
  } else if (amax_out != nullptr) {
    if (cudaMemsetAsync(amax_out, 0, sizeof(float), st) != cudaSuccess) return record_cuda(cudaGetLastError());
  }
  if (rows * cols == 0 && scale_inv_out == nullptr) return TE_OK;
  // An empty tensor still launches one (load-free) tile so that scale_inv_out is published.
  Fp8Args a{rows, cols, scale, amax_out, compute_scale, fmt == TE_E4M3 ? 448.0f : 57344.0f, q_row, q_col,
            compute_scale ? nullptr : amax_out, scale_inv_out};
  const dim3 grid = rows * cols == 0 ? dim3(1, 1) : tile_grid(rows, cols);
  if (in_dtype == TE_BF16) {
    const auto* p = static_cast<const __nv_bfloat16*>(x);
    if (fmt == TE_E4M3) fp8_kernel<__nv_bfloat16, false><<<grid, kThreads, 0, st>>>(p, a);
    else fp8_kernel<__nv_bfloat16, true><<<grid, kThreads, 0, st>>>(p, a);
  } else {
    const auto* p = static_cast<const float*>(x);
    if (fmt == TE_E4M3) fp8_kernel<float, false><<<grid, kThreads, 0, st>>>(p, a);
    else fp8_kernel<float, true><<<grid, kThreads, 0, st>>>(p, a);
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
  if (!grid_ok(rows)) return TE_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (q_row && (s = zero_scales(s_row, TE_E8M0, rows, cols, st)) != TE_OK) return s;
  if (q_col && (s = zero_scales(s_col, TE_E8M0, cols, rows, st)) != TE_OK) return s;
  if (rows * cols == 0 || (!q_row && !q_col)) return TE_OK;
  MxArgs a{rows, cols, q_row, s_row, kpad_of(TE_E8M0, cols), q_col, s_col, kpad_of(TE_E8M0, rows)};
  const dim3 grid = tile_grid(rows, cols);
  if (in_dtype == TE_BF16) mxfp8_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(x), a);
  else mxfp8_kernel<float><<<grid, kThreads, 0, st>>>(static_cast<const float*>(x), a);
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
  if (rows * cols >= (int64_t(1) << 34) || !grid_ok(rows)) return TE_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (row && (s = zero_scales(s_row, TE_UE4M3, rows, cols, st)) != TE_OK) return s;
  if (col && (s = zero_scales(s_col, TE_UE4M3, cols, rows, st)) != TE_OK) return s;
  if (rows * cols == 0 || (!row && !col)) return TE_OK;
  NvArgs a{rows, cols, flags, rht_signs & 0xFFFFu,
           static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32),
           static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32),
           amax, amax_rht, q_row, s_row, gdec_row, kpad_of(TE_UE4M3, cols),
           q_col, s_col, gdec_col, kpad_of(TE_UE4M3, rows)};
  const dim3 grid = tile_grid(rows, cols);
  if (in_dtype == TE_BF16) nvfp4_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(x), a);
  else nvfp4_kernel<float><<<grid, kThreads, 0, st>>>(static_cast<const float*>(x), a);
  count_launch();
  return launch_status();
}

}  // extern "C"
