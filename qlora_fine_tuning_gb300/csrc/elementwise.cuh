// elementwise.cuh -- HBM-bound kernels of the QLoRA linear path:
//   * 4-bit -> bf16 (and fp32) dequantisation, row-major and transposed
//   * 4-bit quantisation of a fp32 / bf16 weight (the stored form)
//   * small transposes and deterministic reductions of split partial sums,
//     used by the single-CTA fallback and the static-scratch XA entry point
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace qlora {

// deq(W)[n,k] = bf16( fp32( codebook[code(n,k)] * absmax[(n*K+k)/64] ) ).
// code(n,k) is the low nibble of byte (n*K+k)/2 for even k, the high nibble
// for odd k.  The fp32 product uses __fmul_rn (IEEE, subnormals kept) and
// the bf16 rounding is round-to-nearest-even.
//
// A group is 8 consecutive weights: one 32-bit word of 4 packed bytes, one
// absmax (8 weights never straddle a 64-block), one 16-byte bf16 store (and
// two 16-byte fp32 stores when requested).  A warp takes chunks of 4 x 32
// consecutive groups; lane l converts groups l, 32+l, 64+l, 96+l of its
// chunk, issuing the four loads before any arithmetic so that four are in
// flight, and each of its stores is one contiguous 512-byte warp store.
__device__ __forceinline__ void dequant_group(uint32_t packed, float am, const float* cb, int64_t g,
                                              uint4* __restrict__ out_bf16, float4* __restrict__ out_f32) {
  float w[8];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t byte = (packed >> (8 * b)) & 0xFFu;
    w[2 * b] = __fmul_rn(cb[byte & 0xFu], am);
    w[2 * b + 1] = __fmul_rn(cb[byte >> 4], am);
  }
  if (out_bf16) {
    uint4 o;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(w[0], w[1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(w[2], w[3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(w[4], w[5]);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(w[6], w[7]);
    o.x = *reinterpret_cast<uint32_t*>(&h0);
    o.y = *reinterpret_cast<uint32_t*>(&h1);
    o.z = *reinterpret_cast<uint32_t*>(&h2);
    o.w = *reinterpret_cast<uint32_t*>(&h3);
    out_bf16[g] = o;
  }
  if (out_f32) {
    out_f32[2 * g] = make_float4(w[0], w[1], w[2], w[3]);
    out_f32[2 * g + 1] = make_float4(w[4], w[5], w[6], w[7]);
  }
}

__global__ void __launch_bounds__(256) dequant4_kernel(const uint32_t* __restrict__ idx4,
                                                       const float* __restrict__ absmax,
                                                       const float* __restrict__ codebook, int64_t n_groups,
                                                       uint4* __restrict__ out_bf16,
                                                       float4* __restrict__ out_f32) {
  __shared__ float cb[16];
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x < 16) cb[threadIdx.x] = codebook[threadIdx.x];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t chunks = (n_groups + 127) / 128;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); c < chunks;
       c += warps) {
    const int64_t g0 = c * 128 + lane;
    uint32_t packed[4];
    float am[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t g = g0 + 32 * i;
      packed[i] = g < n_groups ? __ldg(idx4 + g) : 0u;
      am[i] = g < n_groups ? __ldg(absmax + (g >> 3)) : 0.f;  // 8 groups per 64-block
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t g = g0 + 32 * i;
      if (g < n_groups) dequant_group(packed[i], am[i], cb, g, out_bf16, out_f32);
    }
  }
}

// 4-bit quantisation (the storage the path starts from; the pages load their
// models with load_in_4bit=True -- "利用 Unsloth 和 NVIDIA 硬件加速 LLM 训练",
// section 代码实战):
// absmax = max |w| over each 64-block of the row-major flattening; the code
// of an element is the first i minimising |t - codebook[i]|, t = w / absmax
// as a double division (t = 0 for a zero block) and each distance a double
// subtraction.  The codebook need not be sorted.
//
// The decision is made in fp32 first and confirmed in double only when fp32
// cannot settle it (|t| <= 1 throughout):
//  * sorted codebook: the code is the number of midpoints (c_i + c_{i+1})/2
//    below t.  t32 = w * (1/absmax) (a correctly rounded division when
//    absmax is tiny) is within 2^-22 of t and each fp32
//    midpoint within 2^-24 max|c| of the exact one, so when t32 is farther
//    than `margin` from both neighbouring midpoints, t lies strictly inside
//    the same cell and the double argmin is that code, uniquely.
//  * any codebook: a scan of the 16 fp32 distances (t32 = w / absmax,
//    correctly rounded); every fp32 distance is within 2^-23 (1 + max|c|) of
//    its double counterpart, so a best-vs-runner-up gap above `margin`
//    settles the double argmin too.
// Otherwise (ties, near ties -- rare) the 16 distances are recomputed in
// double: exactly the definition.  In the sorted case a per-CTA table over
// t settles almost every element with one shared-memory byte; elements in
// the few buckets next to a midpoint take a branch-free binary search.  Eight lanes share a block: each converts
// 8 consecutive weights (one 32-byte fp32 or 16-byte bf16 load), absmax is a
// max over the 8 lanes, each lane writes its 4 packed bytes and the block's
// first lane its absmax.
__device__ __forceinline__ int quant_code_exact(float v, float am, const double* cb64) {
  const double t = (am == 0.f) ? 0.0 : __ddiv_rn(static_cast<double>(v), static_cast<double>(am));
  double db = 0.0;
  int code = 0;
  for (int i = 0; i < 16; ++i) {
    const double d = fabs(__dsub_rn(t, cb64[i]));
    if (i == 0 || d < db) {
      db = d;
      code = i;
    }
  }
  return code;
}

constexpr int kQuantBuckets = 16384;            // buckets of width 2/16384 over t in [-1, 1]
constexpr int kQuantLut = kQuantBuckets + 16;    // entries 0..16384, padded
constexpr float kQuantBias = 8396800.0f;         // 2^23 + 8192: fl(x + kQuantBias) has x rounded in its low bits

__device__ __forceinline__ uint32_t bfi4(uint32_t field, uint32_t word, uint32_t pos) {
  uint32_t d;
  asm("bfi.b32 %0, %1, %2, %3, 4;" : "=r"(d) : "r"(field), "r"(word), "r"(pos));
  return d;
}

// Sorted codebook, t32 next to a midpoint (its table bucket is not clear):
// the number of midpoints below t32 by a branch-free binary search, confirmed
// in double when t32 is within `margin` of a midpoint.  Out of line: a few
// elements in a thousand come here, and the warp's main loop stays short.
__device__ __noinline__ int quant_code_near(float t32, float v, float am, const float* mid, const double* cb64,
                                            float margin) {
  int code = (t32 > mid[7]) ? 8 : 0;
  code += (t32 > mid[code + 3]) ? 4 : 0;
  code += (t32 > mid[code + 1]) ? 2 : 0;
  code += (t32 > mid[code]) ? 1 : 0;
  const float lo = code > 0 ? fabsf(__fsub_rn(t32, mid[max(code - 1, 0)])) : INFINITY;
  const float hi = code < 15 ? fabsf(__fsub_rn(mid[min(code, 14)], t32)) : INFINITY;
  if (!(fminf(lo, hi) > margin)) code = quant_code_exact(v, am, cb64);
  return code;
}

// Sorted codebook, absmax outside the range where the scaled reciprocal is
// a normal float (or zero): the eight codes of a group by correctly rounded
// division.
__device__ __noinline__ uint32_t quant_group_divide(const float* v, float am, const float* mid, const double* cb64,
                                                    float margin) {
  uint32_t packed = 0;
  for (int j = 0; j < 8; ++j) {
    const float t32 = (am == 0.f) ? 0.f : __fdiv_rn(v[j], am);
    packed = bfi4(static_cast<uint32_t>(quant_code_near(t32, v[j], am, mid, cb64, margin)), packed, 4u * j);
  }
  return packed;
}

template <bool BF16_IN>
__global__ void __launch_bounds__(1024, 1) quantize4_kernel(const void* __restrict__ w,
                                                        const float* __restrict__ codebook, int64_t n_groups,
                                                        uint32_t* __restrict__ idx4, float* __restrict__ absmax) {
  __shared__ float cb[16];
  __shared__ float mid[15];
  __shared__ double cb64[16];
  __shared__ int8_t lut[kQuantLut];
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x < 16) {
    cb[threadIdx.x] = codebook[threadIdx.x];
    cb64[threadIdx.x] = static_cast<double>(codebook[threadIdx.x]);
  }
  __syncthreads();
  if (threadIdx.x < 15) mid[threadIdx.x] = __fmul_rn(__fadd_rn(cb[threadIdx.x], cb[threadIdx.x + 1]), 0.5f);
  __syncthreads();
  float cmax = 0.f;
  bool sorted = true;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    cmax = fmaxf(cmax, fabsf(cb[i]));
    if (i > 0 && !(cb[i - 1] < cb[i])) sorted = false;
  }
  const float margin = 1.0e-6f * (1.0f + cmax);
  const int lane = threadIdx.x & 31;
  const unsigned grp_mask = 0xFFu << (lane & 24);  // the 8 lanes of this block
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;  // a multiple of 8
  // Software pipelined: the next group's load is issued before the current
  // group is converted, so two loads per thread are in flight.
  auto load8 = [&](int64_t g, float (&v)[8]) {
    if (BF16_IN) {
      const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(w) + g);  // read once: streaming
      const uint32_t q4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(q4[j] << 16);
        v[2 * j + 1] = __uint_as_float(q4[j] & 0xFFFF0000u);
      }
    } else {
      const float4 a = __ldcs(reinterpret_cast<const float4*>(w) + 2 * g);  // read once: streaming
      const float4 b = __ldcs(reinterpret_cast<const float4*>(w) + 2 * g + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
  };
  int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  float nx[8];
  if (g < n_groups) load8(g, nx);  // in flight while the table is built
  // Sorted codebook: bucket j (0..16384) covers t in [-1 + (j - 1/2) h,
  // -1 + (j + 1/2) h), h = 2/16384.  The kernel takes j as the low bits of
  // xb = fl(v * s8 + 2^23 + 8192), s8 = 8192 fl(1/am) (exact scaling): in
  // [2^23, 2^24) the float grid is the integers, so xb is 8192 t' + 8192
  // rounded to an integer, with t' = t (1 + d), |d| <= 2^-24 (the rounding
  // of 1/am), t = v/am exact, |t| <= 1.  So 8192 t' is within 2^-11 of
  // 8192 t, and the bucket found is t's own or a neighbour when t lies within
  // 2^-11 / 8192 < 6.1e-8 of its edge.  Entry of a bucket, with its range
  // widened by 2*margin on both sides (which covers that 6.1e-8):
  //   k >= 0   no fp32 midpoint in the range: every t that can land here has
  //            k midpoints below it, so code k, with the margin to spare;
  //   ~k < 0   exactly one, midpoint k: code k + (t32 > mid[k]), settled in
  //            fp32 when |t32 - mid[k]| > margin, else in double;
  //   -128     several (a codebook with values closer than the bucket):
  //            quant_code_near decides.
  // Thread t fills buckets t, t + blockDim, ... (neighbouring threads write
  // neighbouring bytes), walking the sorted midpoints once.
  {
    const float h = 2.0f / static_cast<float>(kQuantBuckets);
    int pm = 0;
    for (int b = static_cast<int>(threadIdx.x); b <= kQuantBuckets; b += static_cast<int>(blockDim.x)) {
      const float lo = -1.0f + (static_cast<float>(b) - 0.5f) * h;
      const float hi = lo + h;
      while (pm < 15 && mid[pm] < lo - 2.0f * margin) ++pm;
      int8_t e;
      if (!sorted) e = -128;
      else if (pm == 15 || mid[pm] > hi + 2.0f * margin) e = static_cast<int8_t>(pm);
      else if (pm + 1 < 15 && mid[pm + 1] <= hi + 2.0f * margin) e = -128;
      else e = static_cast<int8_t>(~pm);
      lut[b] = e;
    }
  }
  __syncthreads();
  for (; g < n_groups; g += stride) {
    // n_groups is a multiple of 8 and the 8 lanes of a block start 8-aligned,
    // so the 8 lanes of a block are all active here or all gone.
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = nx[j];
    if (g + stride < n_groups) load8(g + stride, nx);
    float am = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) am = fmaxf(am, fabsf(v[j]));
    am = fmaxf(am, __shfl_xor_sync(grp_mask, am, 1, 8));
    am = fmaxf(am, __shfl_xor_sync(grp_mask, am, 2, 8));
    am = fmaxf(am, __shfl_xor_sync(grp_mask, am, 4, 8));
    uint32_t packed = 0;
    if (sorted) {
      // 8192/absmax is a normal float inside this range; divide outside it
      if (am >= 1.0e-33f && am <= 1.0e33f) {
        const float s8 = __fmul_rn(__frcp_rn(am), 8192.0f);
        int32_t neg = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float xb = __fmaf_rn(v[j], s8, kQuantBias);
          const int32_t code = lut[__float_as_int(xb) - 0x4B000000];
          neg |= code;
          packed = bfi4(static_cast<uint32_t>(code), packed, 4u * j);
        }
        if (neg < 0) {  // an element next to a midpoint (one group in ~70)
          const float inv = __fmul_rn(s8, 1.0f / 8192.0f);  // fl(1/am), exactly
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int32_t e = lut[__float_as_int(__fmaf_rn(v[j], s8, kQuantBias)) - 0x4B000000];
            if (e >= 0) continue;
            const float t32 = __fmul_rn(v[j], inv);
            int code;
            if (e == -128) {
              code = quant_code_near(t32, v[j], am, mid, cb64, margin);
            } else {
              const int k = ~e;
              const float d = __fsub_rn(t32, mid[k]);
              code = k + (d > 0.f ? 1 : 0);
              if (!(fabsf(d) > margin)) code = quant_code_exact(v[j], am, cb64);
            }
            packed = bfi4(static_cast<uint32_t>(code), packed, 4u * j);
          }
        }
      } else {
        float vs[8];  // only this rare branch takes an address (keeps v in registers)
#pragma unroll
        for (int j = 0; j < 8; ++j) vs[j] = v[j];
        packed = quant_group_divide(vs, am, mid, cb64, margin);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float t32 = (am == 0.f) ? 0.f : __fdiv_rn(v[j], am);
        float d1 = INFINITY, d2 = INFINITY;
        int code = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float d = fabsf(__fsub_rn(t32, cb[i]));
          if (d < d1) {
            d2 = d1;
            d1 = d;
            code = i;
          } else if (d < d2) {
            d2 = d;
          }
        }
        if (!(__fsub_rn(d2, d1) > margin)) code = quant_code_exact(v[j], am, cb64);
        packed |= static_cast<uint32_t>(code) << (4 * j);
      }
    }
    idx4[g] = packed;
    if ((lane & 7) == 0) absmax[g >> 3] = am;
  }
}

// Transposed dequantisation: outT[k,n] = deq(W)[n,k], outT is [K, N] with
// row stride ldt elements.  One CTA converts a 64(n) x 64(k) tile through
// shared memory so both the packed reads and the bf16 writes are coalesced.
__global__ void __launch_bounds__(256) dequant4_t_kernel(const uint8_t* __restrict__ idx,
                                                         const float* __restrict__ absmax,
                                                         const float* __restrict__ codebook, int32_t N, int32_t K,
                                                         __nv_bfloat16* __restrict__ outT, int64_t ldt) {
  __shared__ float cb[16];
  __shared__ __nv_bfloat16 tile[64][64 + 2];
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x < 16) cb[threadIdx.x] = codebook[threadIdx.x];
  __syncthreads();
  const int n0 = blockIdx.y * 64;
  const int k0 = blockIdx.x * 64;
  // load: 64 rows x 32 bytes; thread t handles row t/4, bytes (t%4)*8 .. +8
  {
    const int rr = threadIdx.x >> 2;
    const int cb8 = (threadIdx.x & 3) * 8;
    const int n = n0 + rr;
    if (n < N) {
      const int64_t e0 = static_cast<int64_t>(n) * K + k0;
      const uint2 pk = *reinterpret_cast<const uint2*>(idx + e0 / 2 + cb8);
      const float am = absmax[e0 / 64];
      const uint32_t words[2] = {pk.x, pk.y};
#pragma unroll
      for (int wi = 0; wi < 2; ++wi) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint32_t byte = (words[wi] >> (8 * b)) & 0xFFu;
          const int kk = 2 * (cb8 + wi * 4 + b);
          tile[rr][kk] = __float2bfloat16_rn(__fmul_rn(cb[byte & 0xFu], am));
          tile[rr][kk + 1] = __float2bfloat16_rn(__fmul_rn(cb[byte >> 4], am));
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) tile[rr][2 * cb8 + j] = __float2bfloat16_rn(0.f);
    }
  }
  __syncthreads();
  // store: 64 rows (k) x 64 (n); thread t writes k-row t/4, n (t%4)*16 .. +16
  {
    const int kr = threadIdx.x >> 2;
    const int nc = (threadIdx.x & 3) * 16;
    const int k = k0 + kr;
    if (k < K) {
      __nv_bfloat16* dst = outT + static_cast<int64_t>(k) * ldt + n0 + nc;
      if (n0 + nc + 16 <= N) {
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          __nv_bfloat162 h;
          h.x = tile[nc + 2 * j][kr];
          h.y = tile[nc + 2 * j + 1][kr];
          w[j] = *reinterpret_cast<uint32_t*>(&h);
        }
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
      } else {
        for (int j = 0; j < 16 && n0 + nc + j < N; ++j) dst[j] = tile[nc + j][kr];
      }
    }
  }
}

// Up to three small transposes in one launch (blockIdx.z selects the job):
// dst[c, rr] = src[rr, c] for rr < rows, c < cols, and zero where the
// dst_rows x dst_cols destination extends beyond the source (padding).
struct TransposeJob {
  const __nv_bfloat16* src;
  __nv_bfloat16* dst;
  int32_t rows, cols, dst_rows, dst_cols;
  int64_t lds, ldd;
  int32_t tiles_x;      // 32-wide tiles over dst_cols
  int32_t tile_begin;   // first flat tile index of this job
};
struct TransposeJobs {
  TransposeJob job[3];
  int32_t njobs;
};

// Flat grid: block b belongs to the last job whose tile_begin <= b.
__global__ void __launch_bounds__(256) transpose_jobs_kernel(const TransposeJobs jobs) {
  __shared__ __nv_bfloat16 t[32][34];
  griddep_wait();
  griddep_launch_dependents();
  int j = 0;
  for (int q = 1; q < jobs.njobs; ++q)
    if (static_cast<int>(blockIdx.x) >= jobs.job[q].tile_begin) j = q;
  const TransposeJob& jb = jobs.job[j];
  const int local = static_cast<int>(blockIdx.x) - jb.tile_begin;
  const int r0 = (local % jb.tiles_x) * 32;  // src rows = dst cols
  const int c0 = (local / jb.tiles_x) * 32;  // src cols = dst rows
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int i = ty; i < 32; i += 8) {
    const int rr = r0 + i, c = c0 + tx;
    t[i][tx] = (rr < jb.rows && c < jb.cols) ? jb.src[static_cast<int64_t>(rr) * jb.lds + c] : __float2bfloat16_rn(0.f);
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int dr = c0 + i, dc = r0 + tx;
    if (dr < jb.dst_rows && dc < jb.dst_cols) jb.dst[static_cast<int64_t>(dr) * jb.ldd + dc] = t[tx][i];
  }
}

// Sum of `splits` fp32 partials P[s][i][j] (i < rows, j < cols, row stride ld,
// split stride sstride), in split order.  Writes any of:
//   out_bf16[i][j]   = bf16(sum)            (ld_o)
//   out_bf16_s[i][j] = bf16(scale * sum)    (ld_o)
//   out_bf16_t[j][i] = bf16(sum)            (ld_t)
//   out_f32[i][j]    = scale * sum          (ld_o)
//   out_f32_t[j][i]  = scale * sum          (ld_t)
// One CTA reduces a 32 x 32 tile; the transposed outputs go through shared
// memory so every global access is coalesced.
struct ReduceArgs {
  const float* part;
  int32_t splits, rows, cols;
  int64_t ld, sstride;
  float scale;
  __nv_bfloat16* out_bf16;
  __nv_bfloat16* out_bf16_s;
  __nv_bfloat16* out_bf16_t;
  float* out_f32;
  float* out_f32_t;
  int64_t ld_o, ld_t;
};

__global__ void __launch_bounds__(256) reduce_tile_kernel(const ReduceArgs a) {
  __shared__ float t[32][33];
  griddep_wait();
  griddep_launch_dependents();
  const int r0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int c = c0 + tx;
  for (int i = ty; i < 32; i += 8) {
    const int r = r0 + i;
    float acc = 0.f;
    if (r < a.rows && c < a.cols) {
      const float* pp = a.part + static_cast<int64_t>(r) * a.ld + c;
      for (int s = 0; s < a.splits; ++s) acc += pp[s * a.sstride];
      const int64_t o = static_cast<int64_t>(r) * a.ld_o + c;
      if (a.out_bf16) a.out_bf16[o] = __float2bfloat16_rn(acc);
      if (a.out_bf16_s) a.out_bf16_s[o] = __float2bfloat16_rn(__fmul_rn(a.scale, acc));
      if (a.out_f32) a.out_f32[o] = __fmul_rn(a.scale, acc);
    }
    t[i][tx] = acc;
  }
  if (!a.out_bf16_t && !a.out_f32_t) return;
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int cc = c0 + i, r = r0 + tx;
    if (cc < a.cols && r < a.rows) {
      const float v = t[tx][i];
      const int64_t o = static_cast<int64_t>(cc) * a.ld_t + r;
      if (a.out_bf16_t) a.out_bf16_t[o] = __float2bfloat16_rn(v);
      if (a.out_f32_t) a.out_f32_t[o] = __fmul_rn(a.scale, v);
    }
  }
}

}  // namespace qlora
