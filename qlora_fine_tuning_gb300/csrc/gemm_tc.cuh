// gemm_tc.cuh -- persistent tcgen05 / TMEM / TMA GEMM for sm_103a.
//
// D[128-row tile, bn-col tile] = sum_red A[row, red] * B[col, red]
//   (+ optional rank-r "LoRA" K-steps A2[row, :] * B2[col, :] into the same
//    TMEM accumulator).
//
// Every contraction of the QLoRA linear layer is an instance:
//   XA  = X . A            (A-op X K-major, B-op A^T)          fp32 split-K partials
//   Y   = X . Wd^T + (s XA) . B    (B-op Wd; LoRA: A2 = s*XA, B2 = B^T)  bf16
//   G   = dY . B^T per adapter segment                         fp32 split partials
//   dX  = dY . Wd + (s G) . A^T    (B-op Wd^T; LoRA: A2 = s*G, B2 = A)  bf16
//   dA  = X^T . G          (A-op X read MN-major, B-op G^T)    fp32 split partials
//   dB^T= dY^T . XA        (A-op dY read MN-major, B-op XA^T)  fp32 split partials
//
// Persistent: each CTA walks the tile list (row tile fastest, then column
// tile, then split/segment) with stride gridDim.x.  Roles (6 warps):
//   warp 0 lane 0  TMA producer, runs ahead across tile boundaries through a
//                  ring of `stages` shared-memory stages;
//   warp 1         MMA issuer: tcgen05.mma (M=128, N=bn, K=16) into one of two
//                  TMEM accumulators (tile j uses buffer j&1);
//   warps 2..5     epilogue: tcgen05.ld of the finished accumulator, convert,
//                  store; then release the buffer -- so the epilogue of tile j
//                  overlaps the mainloop of tile j+1.
// Warp 0 owns the TMEM allocation (2 x bn columns rounded to a power of two).
//
// Shared-memory tiles use the 128-byte swizzle written by TMA:
//   K-major operand  : row i at i*128 B holds 64 reduction elements; 8-row
//                      atoms of 1024 B (SBO = 1024); a 16-wide K step is +32 B.
//   MN-major operand : row j at j*128 B holds 64 output-index elements for
//                      reduction index j; 8-row atoms (SBO = 1024); the second
//                      64-wide output block sits 8192 B further (LBO);
//                      a 16-wide K step is +2048 B.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace qlora {

enum GemmMode : int32_t {
  GM_PLAIN = 0,  // no segments, no LoRA steps
  GM_FWD = 1,    // LoRA steps; adapter segment chosen by the output-column tile
  GM_G = 2,      // segment = z / splits; reduction over that segment's columns
  GM_DX = 3,     // LoRA steps over all segments at once
  GM_DB = 4,     // segment chosen by the output-row tile; B rows offset by seg*r
};

constexpr int kMaxSeg = 8;
constexpr int kMaxStages = 8;
constexpr uint32_t kATileBytes = 128 * 128;  // 128 rows x 64 bf16

struct GemmArgs {
  int32_t M;          // output rows (masking)
  int32_t N;          // output cols (masking, before out_col0)
  int32_t bn;         // tile width = UMMA N (16..256, multiple of 16)
  int32_t stages;     // ring depth (<= kMaxStages)
  uint32_t stage_bytes;
  int32_t mode;
  int32_t red_len;    // reduction length in elements (modes other than GM_G)
  int32_t splits;     // reduction splits (z % splits)
  int32_t r;          // adapter rank
  int32_t nseg;
  int32_t seg_start[kMaxSeg + 1];  // segment boundaries over the layer's N
  int32_t lora_atoms;   // number of 64-wide LoRA K blocks (0..4)
  int32_t lora_ksteps;  // number of 16-wide LoRA K steps in total
  int32_t out_ld;       // output row stride in elements
  int32_t out_valid;    // columns n0+c >= out_valid are not stored
  int64_t out_split_stride;  // elements between split partial outputs
  int32_t m_tiles, n_tiles, z_tiles;  // tile grid (row tiles fastest)
  void* out;
  uint32_t* err;        // device error word (bit flags), may be null
  uint64_t timeout_ns;  // bound on every barrier wait
  int32_t debug_stall;  // test hook: CTA (pair) 0 never fills its first stage
  int32_t l2_hints;     // bit 0: streaming (evict-first) output stores;
                        // bit 1: A loads evict-last; bit 2: B loads evict-first
  const float* codebook;  // 16 fp32 values (pair kernel with in-kernel dequantisation)
  int32_t dq_k;           // K of the 4-bit weight (pair kernel with in-kernel dequantisation)
};

struct TileInfo {
  int m0, n0, split, red_begin, kb0, n_main, n_iter, b_row0, a2_x0, out_col0;
};

__device__ __forceinline__ int seg_index(const GemmArgs& p, int pos) {
  int sg = 0;
#pragma unroll 1
  for (int j = 1; j < p.nseg; ++j)
    if (pos >= p.seg_start[j]) sg = j;
  return sg;
}

// Everything a role needs to know about one tile; all roles derive it the
// same way from the tile index.
__device__ __forceinline__ TileInfo tile_info(const GemmArgs& p, int tile) {
  TileInfo t;
  const int mt = tile % p.m_tiles;
  const int rest = tile / p.m_tiles;
  const int nt = rest % p.n_tiles;
  const int z = rest / p.n_tiles;
  t.m0 = mt * 128;
  t.n0 = nt * p.bn;
  t.split = z % p.splits;
  int sg = 0;
  if (p.mode == GM_FWD) sg = seg_index(p, t.n0);
  else if (p.mode == GM_DB) sg = seg_index(p, t.m0);
  else if (p.mode == GM_G) sg = z / p.splits;
  int red_end = p.red_len;
  t.red_begin = 0;
  if (p.mode == GM_G) {
    t.red_begin = p.seg_start[sg];
    red_end = p.seg_start[sg + 1];
  }
  const int nkb = (red_end - t.red_begin + 63) / 64;
  const int chunk = (nkb + p.splits - 1) / p.splits;
  t.kb0 = min(nkb, t.split * chunk);
  t.n_main = min(nkb, t.kb0 + chunk) - t.kb0;
  const bool has_lora = (p.mode == GM_FWD || p.mode == GM_DX) && p.lora_atoms > 0;
  t.n_iter = t.n_main + (has_lora ? p.lora_atoms : 0);
  t.b_row0 = t.n0 + (p.mode == GM_DB ? sg * p.r : 0);
  t.a2_x0 = (p.mode == GM_FWD ? sg * p.r : 0);
  t.out_col0 = (p.mode == GM_G ? sg * p.r : 0);
  return t;
}

__device__ __forceinline__ void report(const GemmArgs& p, uint32_t bit) {
  if (p.err) atomicOr(p.err, bit);
}

// Bounded wait that also gives up as soon as another role raised `abort`.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <bool A_MN, bool OUT_F32>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                   const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((((raw + 1023u) & ~1023u)) - raw);
  uint8_t* ctrl = smem + static_cast<uint32_t>(p.stages) * p.stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;   // [2] accumulator ready
  uint64_t* tempty = tfull + 2;           // [2] accumulator drained
  uint64_t* mma_done = tempty + 2;        // every MMA of this CTA completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total = p.m_tiles * p.n_tiles * p.z_tiles;
  const bool has_lora = (p.mode == GM_FWD || p.mode == GM_DX) && p.lora_atoms > 0;
  uint32_t acc_cols = 32;
  while (acc_cols < static_cast<uint32_t>(p.bn)) acc_cols <<= 1;
  const uint32_t tmem_cols = 2 * acc_cols;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  if (warp == 1 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (has_lora) {
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above touched only on-chip state; global memory written by the
  // predecessor kernel is visible after this point.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ---------------- TMA producer (whole warp, one elected lane issues) ----------------
    const uint32_t tx = kATileBytes + static_cast<uint32_t>(p.bn) * 128u;
    uint32_t g = 0;  // iterations issued so far (ring position)
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const TileInfo t = tile_info(p, tile);
      for (int it = 0; it < t.n_iter; ++it) {
        const uint32_t s = g % static_cast<uint32_t>(p.stages);
        const uint32_t ph = (g / static_cast<uint32_t>(p.stages)) & 1u;
        if (!warp_wait(&empty[s], ph ^ 1u, p.timeout_ns, abort_flag)) {
          if (lane == 0) {
            if (!*abort_flag) report(p, 1u);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
        if (p.debug_stall && g == 0 && blockIdx.x == 0) {  // leave stage 0 empty: its consumer times out
          ++g;
          continue;
        }
        uint8_t* a_dst = smem + s * p.stage_bytes;
        uint8_t* b_dst = a_dst + kATileBytes;
        mbar_arrive_expect_tx_ws(&full[s], tx);
        if (it < t.n_main) {
          const int kel = t.red_begin + (t.kb0 + it) * 64;
          if (A_MN) {
            tma_load_2d_ws(a_dst, &tmA, &full[s], t.m0, kel);
            tma_load_2d_ws(a_dst + 8192, &tmA, &full[s], t.m0 + 64, kel);
          } else {
            tma_load_2d_ws(a_dst, &tmA, &full[s], kel, t.m0);
          }
          tma_load_2d_ws(b_dst, &tmB, &full[s], kel, t.b_row0);
        } else {
          const int a = it - t.n_main;
          tma_load_2d_ws(a_dst, &tmA2, &full[s], t.a2_x0 + 64 * a, t.m0);
          tma_load_2d_ws(b_dst, &tmB2, &full[s], 64 * a, t.n0);
        }
        ++g;
      }
    }
    // Do not leave the CTA while copies it issued may still land in smem.
    if (lane == 0) {
      const uint32_t S = static_cast<uint32_t>(p.stages);
      for (uint32_t q = (g > S ? g - S : 0u); q < g; ++q) mbar_wait(&full[q % S], (q / S) & 1u, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
    const uint32_t idesc_main = idesc_bf16_f32(128, static_cast<uint32_t>(p.bn), A_MN, false);
    const uint32_t idesc_lora = idesc_bf16_f32(128, static_cast<uint32_t>(p.bn), false, false);
    const uint64_t a_step = A_MN ? (2048u >> 4) : (32u >> 4);
    uint32_t g = 0;
    int j = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++j) {
      const TileInfo t = tile_info(p, tile);
      const uint32_t acc = static_cast<uint32_t>(j & 1);
      if (!warp_wait(&tempty[acc], (static_cast<uint32_t>(j >> 1) & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
        if (lane == 0) {
          if (!*abort_flag) report(p, 8u);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * acc_cols;
      for (int it = 0; it < t.n_iter; ++it) {
        const uint32_t s = g % static_cast<uint32_t>(p.stages);
        const uint32_t ph = (g / static_cast<uint32_t>(p.stages)) & 1u;
        if (!warp_wait(&full[s], ph, p.timeout_ns, abort_flag)) {
          if (lane == 0) {
            if (!*abort_flag) report(p, 2u);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + s * p.stage_bytes);
        const uint32_t b_addr = a_addr + kATileBytes;
        if (it < t.n_main) {
          const uint64_t ad = A_MN ? sdesc_sw128(a_addr, 8192u, 1024u) : sdesc_sw128(a_addr, 16u, 1024u);
          tc_mma_bf16_k64_ws(d_tmem, ad, sdesc_sw128(b_addr, 16u, 1024u), a_step, 2u, idesc_main,
                             it > 0 ? 1u : 0u);
        } else {
          const int ksteps = min(4, p.lora_ksteps - 4 * (it - t.n_main));
          for (int kk = 0; kk < ksteps; ++kk)
            tc_mma_bf16_ws(d_tmem, sdesc_sw128(a_addr + static_cast<uint32_t>(kk) * 32u, 16u, 1024u),
                           sdesc_sw128(b_addr + static_cast<uint32_t>(kk) * 32u, 16u, 1024u), idesc_lora,
                           (it > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit_ws(&empty[s]);
        ++g;
      }
      if (!ok) break;
      tc_commit_ws(&tfull[acc]);  // arrives once this tile's MMAs have completed
    }
    tc_commit_ws(mma_done);
  } else if (warp >= 2) {
    // ---------------- Epilogue ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    int j = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++j) {
      const TileInfo t = tile_info(p, tile);
      const uint32_t acc = static_cast<uint32_t>(j & 1);
      if (!warp_wait(&tfull[acc], static_cast<uint32_t>(j >> 1) & 1u, p.timeout_ns, abort_flag)) {
        if (lane == 0) {
          if (!*abort_flag) report(p, 4u);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const int grow = t.m0 + row;
      const bool row_ok = grow < p.M;
      const bool have_acc = t.n_iter > 0;
      const uint32_t t_base = tmem_base + acc * acc_cols + (static_cast<uint32_t>(q * 32) << 16);
      const int nchunks = p.bn / 16;
      for (int c = 0; c < nchunks; ++c) {
        uint32_t v[16];
        if (have_acc) {
          tmem_ld16(t_base + static_cast<uint32_t>(c * 16), v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0u;
        }
        const int c0 = t.n0 + c * 16;
        if (!row_ok) continue;
        if (OUT_F32) {
          float* out = reinterpret_cast<float*>(p.out) + static_cast<int64_t>(t.split) * p.out_split_stride +
                       static_cast<int64_t>(grow) * p.out_ld + t.out_col0;
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {
            const int col = c0 + gq * 4;
            if (col < p.out_valid && col < p.N)
              *reinterpret_cast<uint4*>(out + col) =
                  make_uint4(v[gq * 4 + 0], v[gq * 4 + 1], v[gq * 4 + 2], v[gq * 4 + 3]);
          }
        } else {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(grow) * p.out_ld;
#pragma unroll
          for (int gq = 0; gq < 2; ++gq) {
            const int col = c0 + gq * 8;
            if (col < p.out_valid && col < p.N) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(v[gq * 8 + 0]), __uint_as_float(v[gq * 8 + 1]));
              w.y = pack_bf16x2(__uint_as_float(v[gq * 8 + 2]), __uint_as_float(v[gq * 8 + 3]));
              w.z = pack_bf16x2(__uint_as_float(v[gq * 8 + 4]), __uint_as_float(v[gq * 8 + 5]));
              w.w = pack_bf16x2(__uint_as_float(v[gq * 8 + 6]), __uint_as_float(v[gq * 8 + 7]));
              if (p.l2_hints & 1) __stcs(reinterpret_cast<uint4*>(out + col), w);
              else *reinterpret_cast<uint4*>(out + col) = w;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    // mma_done fires only after every MMA this CTA issued has completed, so
    // the allocation is never released under a running MMA.
    if (lane == 0) mbar_wait(mma_done, 0u, p.timeout_ns);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace qlora
