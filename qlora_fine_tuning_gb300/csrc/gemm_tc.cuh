// gemm_tc.cuh -- persistent tcgen05 / TMEM / TMA GEMM for sm_103a.
//
// D[128-row tile, bn-col tile] = sum_red A[row, red] * B[col, red]
//   (+ optional rank-r "LoRA" K-steps A2[row, :] * B2[col, :] into the same
//    TMEM accumulator).
//
// The rank-r contractions of the QLoRA linear layer are instances whose
// reduction splits are summed inside the kernel (EPI_RED, below):
//   XA  = X . A            (A-op X K-major, B-op A read MN-major)   -> XA, s*XA
//   G   = dY . B^T per adapter segment (B-op B K-major)           -> s*G, G
//   dA  = s X^T G          (A-op X read MN-major, B-op G MN-major)  -> dA fp32
//   dB^T= s dY^T . XA      (A-op dY read MN-major, B-op XA MN-major) -> dB fp32
// and, when the CTA-pair kernel cannot be used, the two large products
//   Y   = X . Wd^T + (s XA) . B    (B-op Wd; LoRA: A2 = s*XA, B2 = B^T)  bf16
//   dX  = dY . Wd + (s G) . A^T    (B-op Wd^T; LoRA: A2 = s*G, B2 = A)  bf16
//
// Persistent: each CTA (or cluster, EPI_RED) walks the tile list (row tile
// fastest, then column tile, then segment) with a fixed stride.  Roles
// (6 warps):
//   warp 0         TMA producer, runs ahead across tile boundaries through a
//                  ring of `stages` shared-memory stages;
//   warp 1         MMA issuer: tcgen05.mma (M=128, N=bn, K=16) into one of two
//                  TMEM accumulators (tile j uses buffer j&1);
//   warps 2..5     epilogue: tcgen05.ld of the finished accumulator, convert,
//                  store; then release the buffer -- so the epilogue of tile j
//                  overlaps the mainloop of tile j+1.
// Warp 0 owns the TMEM allocation (2 x bn columns rounded to a power of two).
//
// EPI_RED: the `splits` CTAs that share one output tile form a thread-block
// cluster; CTA k reduces over the k-th chunk of the reduction.  Each CTA
// copies its fp32 accumulator to a shared-memory buffer, then sums one slice
// of the tile's rows over all buffers of the cluster (distributed shared
// memory), in split order 0, 1, ..., so the result does not depend on timing,
// and writes the outputs.  Two mbarriers per CTA pace the exchange: red_ready
// (every CTA's buffer of this round is written) and red_free (every CTA has
// read this CTA's buffer).  No partial sums go through global memory.
//
// Shared-memory tiles use the 128-byte swizzle written by TMA:
//   K-major operand  : row i at i*128 B holds 64 reduction elements; 8-row
//                      atoms of 1024 B (SBO = 1024); a 16-wide K step is +32 B.
//   MN-major operand : row j at j*128 B holds 64 output-index elements for
//                      reduction index j; 8-row atoms (SBO = 1024); the next
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

enum GemmEpi : int {
  EPI_BF16 = 0,      // bf16 output tile
  EPI_F32_PART = 1,  // fp32 partial sum per split (summed by a separate kernel)
  EPI_RED = 2,       // splits summed in the kernel across a cluster
};

constexpr int kMaxSeg = 8;
constexpr uint32_t kRedLd = 68;                     // floats per row of the reduction buffer (64 + 4 pad)
constexpr uint32_t kRedBytes = 128u * kRedLd * 4u;  // one 128 x 64 fp32 chunk
constexpr int kMaxStages = 10;
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
  int32_t tile_m;       // output rows per tile: 128, or (K-major A, EPI_RED) a multiple of 8 below it
  void* out;
  uint32_t* err;        // device error word (bit flags), may be null
  uint64_t timeout_ns;  // bound on every barrier wait
  int32_t debug_stall;  // test hook: CTA (pair) 0 never fills its first stage
  int32_t l2_hints;     // bit 0: streaming (evict-first) output stores;
                        // bit 1: the band's operand evict-last; bit 2: the other evict-first
  int32_t group_m;        // pair kernel tile order: >0 row tiles per band, <0 column tiles per band, 0 one band
  // pair kernel with in-kernel dequantisation: the 4-bit weight [N, K]
  const float* codebook;     // 16 fp32 values
  const uint8_t* dq_idx;     // packed codes [N, K/2]
  const float* dq_absmax;    // one scale per 64-block [N, K/64]
  int32_t dq_k;              // K
  // EPI_RED launch that also writes the bf16 Wd (epi_dequant_slice below):
  __nv_bfloat16* dq_out;     // row-major [N, K]
  int64_t dq_words;          // N*K/8 (8 weights each); 0 = no dequantisation in this launch
  // EPI_RED outputs; `sum` is the full reduction, columns are shifted by out_col0:
  float red_scale;
  __nv_bfloat16* red_bf16;    // sum, row-major [row * red_ld + col]
  __nv_bfloat16* red_bf16_s;  // red_scale * sum, row-major
  float* red_f32;             // red_scale * sum, row-major
  float* red_f32_t;           // red_scale * sum, transposed [col * red_ld_t + row]
  int64_t red_ld, red_ld_t;
  int32_t red_accumulate;     // red_f32 / red_f32_t: add into the existing values instead of overwriting
  int32_t red_in_ring;        // every cluster has one tile: the split-sum buffer reuses ring stage 0
};

// fp32 outputs of the split sum: v, or (accumulate) the existing value plus v.
__device__ __forceinline__ float red_out1(const GemmArgs& p, const float* dst, float v) {
  return p.red_accumulate ? __fadd_rn(*dst, v) : v;
}
__device__ __forceinline__ float4 red_out4(const GemmArgs& p, const float* dst, float4 v) {
  if (!p.red_accumulate) return v;
  const float4 o = *reinterpret_cast<const float4*>(dst);
  return make_float4(__fadd_rn(o.x, v.x), __fadd_rn(o.y, v.y), __fadd_rn(o.z, v.z), __fadd_rn(o.w, v.w));
}

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
  t.m0 = mt * p.tile_m;
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

// Dequantisation carried by a rank-r GEMM launch (XA in the forward, G in the
// backward): while a CTA's producer and MMA warps stream X (or dY), the rest
// of the CTA expands one contiguous slice of the 4-bit weight into the bf16 Wd
// -- six warps whose only work this is, the four epilogue warps until their
// accumulator is ready (and again after the split exchange), and the producer
// and MMA warps once their own work is issued.  Both streams share one launch
// and keep HBM busy together.  The arithmetic is the standalone dequantiser's:
// deq = bf16_rn(fp32(codebook[code] * absmax)) with one __fmul_rn, so Wd is
// the same bit for bit.
// A word is 8 consecutive weights: one 4-byte load of codes, one absmax (8
// words share a 64-block), one 16-byte bf16 store.  A unit is 32 x kDqUnroll
// words, lane l taking words l, l + 32, ..., so that every warp load is 128
// contiguous bytes and every warp store 512; warps claim units from a
// shared-memory counter and load the next unit before converting the current
// one.  Lane l holds codebook[l mod 16] and a lookup is one warp shuffle whose
// source lane is the word shifted to the code (a shuffle reads only the low
// five bits of its lane operand, and lanes l and l + 16 agree); all loop
// bounds are warp-uniform so that every shuffle runs on the full warp.  The
// two products of a byte come from one paired multiply (mul.rn.f32x2, each
// half rounded to nearest like __fmul_rn).
constexpr int kDqUnroll = 16;
struct DqUnit {
  uint32_t c[kDqUnroll];
  float am[kDqUnroll];
};

__device__ __forceinline__ void dq_load(const GemmArgs& p, int64_t base, int64_t w1, int lane, DqUnit& u) {
  const uint32_t* codes = reinterpret_cast<const uint32_t*>(p.dq_idx);
#pragma unroll
  for (int i = 0; i < kDqUnroll; ++i) {
    const int64_t w = base + lane + 32 * i;
    u.c[i] = w < w1 ? __ldg(codes + w) : 0u;
    u.am[i] = w < w1 ? __ldg(p.dq_absmax + (w >> 3)) : 0.f;
  }
}

// bf16 pair (lo, hi) = (bf16_rn(cl * am), bf16_rn(ch * am)); am2 = {am, am}.
__device__ __forceinline__ uint32_t dq_pair(float cl, float ch, uint64_t am2) {
  uint64_t c2, p2;
  asm("mov.b64 %0, {%1, %2};" : "=l"(c2) : "f"(cl), "f"(ch));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p2) : "l"(c2), "l"(am2));
  float f0, f1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f0), "=f"(f1) : "l"(p2));
  return pack_bf16x2(f0, f1);
}

__device__ __forceinline__ void dq_convert(const GemmArgs& p, int64_t base, int64_t w1, int lane, float cbv,
                                           const DqUnit& u) {
  uint4* out = reinterpret_cast<uint4*>(p.dq_out);
#pragma unroll
  for (int i = 0; i < kDqUnroll; ++i) {
    const int64_t w = base + lane + 32 * i;
    uint64_t am2;
    asm("mov.b64 %0, {%1, %1};" : "=l"(am2) : "f"(u.am[i]));
    float c[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) c[k] = __shfl_sync(0xFFFFFFFFu, cbv, static_cast<int>(u.c[i] >> (4 * k)));
    const uint4 o = make_uint4(dq_pair(c[0], c[1], am2), dq_pair(c[2], c[3], am2), dq_pair(c[4], c[5], am2),
                               dq_pair(c[6], c[7], am2));
    if (w < w1) out[w] = o;
  }
}

// One warp's share of this CTA's slice; `ctr` (shared memory, zeroed before
// the roles start) hands out units.  With `poll` (the split-sum warps: the
// barrier of their first accumulator), the warp leaves after the current unit
// once that phase has completed, so that the split exchange runs beside the
// rest of the expansion instead of after it; it calls again afterwards.
__device__ __noinline__ void dq_slice_warp(const GemmArgs& p, uint32_t* ctr, int lane, uint64_t* poll = nullptr) {
  const float cbv = __ldg(p.codebook + (lane & 15));
  const int64_t Wn = p.dq_words;
  const int64_t per = (Wn + gridDim.x - 1) / gridDim.x;
  const int64_t w0 = min(Wn, per * static_cast<int64_t>(blockIdx.x));
  const int64_t w1 = min(Wn, w0 + per);
  const int64_t unit = 32 * kDqUnroll;
  const int64_t units = (w1 - w0 + unit - 1) / unit;
  auto claim = [&]() -> int64_t {
    uint32_t v = 0;
    if (lane == 0) v = atomicAdd(ctr, 1u);
    return static_cast<int64_t>(__shfl_sync(0xFFFFFFFFu, v, 0));
  };
  auto ready = [&]() -> bool {
    if (!poll) return false;
    const bool r = lane == 0 && mbar_try_wait(poll, 0u);
    return __shfl_sync(0xFFFFFFFFu, r ? 1 : 0, 0) != 0;
  };
  if (ready()) return;
  DqUnit cur, nxt;
  int64_t k = claim();
  if (k >= units) return;
  dq_load(p, w0 + k * unit, w1, lane, cur);
  while (true) {
    const int64_t k2 = ready() ? units : claim();
    if (k2 < units) dq_load(p, w0 + k2 * unit, w1, lane, nxt);
    dq_convert(p, w0 + k * unit, w1, lane, cbv, cur);
    if (k2 >= units) break;
    k = k2;
    cur = nxt;
  }
}

// Flat tile index of the T-th tile of a cluster walk (EPI_RED): the cluster
// rank picks the split, z = segment * splits + split.
__device__ __forceinline__ int red_tile(const GemmArgs& p, int T, uint32_t rank) {
  const int mn = p.m_tiles * p.n_tiles;
  return T % mn + mn * ((T / mn) * p.splits + static_cast<int>(rank));
}

// EPI_RED launches carry kRedExtraWarps more warps (6 .. 11) whose only work
// is the Wd slice (none when the launch writes no Wd), so that up to 12 warps
// of a CTA keep code loads in flight.  Measured on the Llama-3-8B MLP step:
// 2 extra warps took 26 us per step off XA + G, 4 and 6 a further 11 and
// 2 us; 10 are slower (the registers a thread may hold fall to 128 and spill).
constexpr int kRedExtraWarps = 6;
constexpr int kRedThreads = 192 + 32 * kRedExtraWarps;

template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(kRedThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ GemmArgs p, const __grid_constant__ GemmArgs p2) {
  constexpr bool RED = (EPI == EPI_RED);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((((raw + 1023u) & ~1023u)) - raw);
  // The split-sum buffer follows the ring, or -- when each cluster takes one
  // tile, so that the ring is idle once that tile's MMAs have completed --
  // occupies the start of the ring itself.
  const bool in_ring = RED && p.red_in_ring;
  float* red = reinterpret_cast<float*>(in_ring ? smem : smem + static_cast<uint32_t>(p.stages) * p.stage_bytes);
  uint8_t* ctrl = smem + static_cast<uint32_t>(p.stages) * p.stage_bytes + ((RED && !in_ring) ? kRedBytes : 0u);
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;   // [2] accumulator ready
  uint64_t* tempty = tfull + 2;           // [2] accumulator drained
  uint64_t* mma_done = tempty + 2;        // every MMA of this CTA completed
  uint64_t* red_ready = mma_done + 1;     // EPI_RED: all buffers of the round written
  uint64_t* red_free = red_ready + 1;     // EPI_RED: this CTA's buffer read by all
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red_free + 1);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);
  uint32_t* dq_ctr = reinterpret_cast<uint32_t*>(tmem_slot + 2);  // units of the Wd slice handed out

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total = p.m_tiles * p.n_tiles * p.z_tiles;
  const int S = RED ? p.splits : 1;
  const uint32_t rank = RED ? cluster_ctarank() : 0u;
  // Tile walk: CTAs (or clusters) take every stride-th tile.
  const int walk_first = RED ? static_cast<int>(blockIdx.x) / S : static_cast<int>(blockIdx.x);
  const int walk_stride = RED ? static_cast<int>(gridDim.x) / S : static_cast<int>(gridDim.x);
  // EPI_RED may carry a second, independent problem `p2` (its own tensor maps
  // in the tmA2 / tmB2 slots, which rank-r GEMMs do not otherwise use): the
  // walk covers p's tiles, then p2's.  p2.m_tiles == 0 means none.
  const int tiles1 = RED ? total / S : total;
  const int tiles2 = RED ? p2.m_tiles * p2.n_tiles * (p2.z_tiles / S) : 0;
  const int walk_total = tiles1 + tiles2;
  const bool has_lora = (p.mode == GM_FWD || p.mode == GM_DX) && p.lora_atoms > 0;
  uint32_t acc_cols = 32;
  while (acc_cols < static_cast<uint32_t>(max(p.bn, tiles2 > 0 ? p2.bn : 0))) acc_cols <<= 1;
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
    if (RED) {
      mbar_init(red_ready, static_cast<uint32_t>(S) * 128u);
      mbar_init(red_free, static_cast<uint32_t>(S) * 128u);
    }
    *abort_flag = 0;
    *dq_ctr = 0u;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  if (warp == 1 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (has_lora || tiles2 > 0) {
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (RED) cluster_sync_all();  // peers' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above touched only on-chip state; global memory written by the
  // predecessor kernel is visible after this point.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ---------------- TMA producer (whole warp, one elected lane issues) ----------------
    uint32_t g = 0;  // iterations issued so far (ring position)
    bool ok = true;
    for (int T = walk_first; T < walk_total && ok; T += walk_stride) {
      const bool second = T >= tiles1;
      const GemmArgs& pq = second ? p2 : p;
      const CUtensorMap* mapA = second ? &tmA2 : &tmA;
      const CUtensorMap* mapB = second ? &tmB2 : &tmB;
      const TileInfo t = tile_info(pq, RED ? red_tile(pq, second ? T - tiles1 : T, rank) : T);
      // A box: tile_m rows of 128 B (rows tile_m..127 of the stage keep stale
      // bytes; they only feed accumulator rows the epilogue never stores).
      const uint32_t tx = static_cast<uint32_t>(pq.tile_m + pq.bn) * 128u;
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
            tma_load_2d_ws(a_dst, mapA, &full[s], t.m0, kel);
            tma_load_2d_ws(a_dst + 8192, mapA, &full[s], t.m0 + 64, kel);
          } else {
            tma_load_2d_ws(a_dst, mapA, &full[s], kel, t.m0);
          }
          if (B_MN) {
            for (int i = 0; i < pq.bn / 64; ++i)
              tma_load_2d_ws(b_dst + i * 8192, mapB, &full[s], t.b_row0 + 64 * i, kel);
          } else {
            tma_load_2d_ws(b_dst, mapB, &full[s], kel, t.b_row0);
          }
        } else {
          const int a = it - t.n_main;
          tma_load_2d_ws(a_dst, &tmA2, &full[s], t.a2_x0 + 64 * a, t.m0);
          tma_load_2d_ws(b_dst, &tmB2, &full[s], 64 * a, t.n0);
        }
        ++g;
      }
    }
    if (RED && p.dq_words > 0) dq_slice_warp(p, dq_ctr, lane);  // every copy is issued: help with Wd
    // Do not leave the CTA while copies it issued may still land in smem.
    if (lane == 0) {
      const uint32_t S_ = static_cast<uint32_t>(p.stages);
      for (uint32_t q = (g > S_ ? g - S_ : 0u); q < g; ++q) mbar_wait(&full[q % S_], (q / S_) & 1u, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
    const uint32_t idesc_lora = idesc_bf16_f32(128, static_cast<uint32_t>(p.bn), false, false);
    const uint64_t a_step = A_MN ? (2048u >> 4) : (32u >> 4);
    const uint64_t b_step = B_MN ? (2048u >> 4) : (32u >> 4);
    uint32_t g = 0;
    int j = 0;
    bool ok = true;
    for (int T = walk_first; T < walk_total && ok; T += walk_stride, ++j) {
      const bool second = T >= tiles1;
      const GemmArgs& pq = second ? p2 : p;
      const TileInfo t = tile_info(pq, RED ? red_tile(pq, second ? T - tiles1 : T, rank) : T);
      const uint32_t idesc_main = idesc_bf16_f32(128, static_cast<uint32_t>(pq.bn), A_MN, B_MN);
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
          const uint64_t bd = B_MN ? sdesc_sw128(b_addr, 8192u, 1024u) : sdesc_sw128(b_addr, 16u, 1024u);
          tc_mma_bf16_k64_ws(d_tmem, ad, bd, a_step, b_step, idesc_main, it > 0 ? 1u : 0u);
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
    if (RED && p.dq_words > 0) dq_slice_warp(p, dq_ctr, lane);  // every MMA is issued: help with Wd
  } else if (warp >= 6) {
    // ---------------- EPI_RED: extra warps, Wd only ----------------
    if (RED && p.dq_words > 0) dq_slice_warp(p, dq_ctr, lane);
  } else if (warp >= 2 && RED) {
    // ---------------- Epilogue: sum the splits across the cluster ----------------
    if constexpr (RED) {
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int et = static_cast<int>(threadIdx.x) - 64;  // 0..127
    if (p.dq_words > 0) dq_slice_warp(p, dq_ctr, lane, &tfull[0]);
    const uint32_t red_s = smem_u32(red);
    const uint32_t ready_s = smem_u32(red_ready);
    const uint32_t free_s = smem_u32(red_free);
    uint32_t round = 0;
    int j = 0;
    bool ok = true;
    for (int T = walk_first; T < walk_total && ok; T += walk_stride, ++j) {
      const bool second = T >= tiles1;
      const GemmArgs& pq = second ? p2 : p;
      const TileInfo t = tile_info(pq, red_tile(pq, second ? T - tiles1 : T, rank));
      const uint32_t acc = static_cast<uint32_t>(j & 1);
      if (!warp_wait(&tfull[acc], static_cast<uint32_t>(j >> 1) & 1u, p.timeout_ns, abort_flag)) {
        if (lane == 0) {
          if (!*abort_flag) report(p, 4u);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const uint32_t t_base = tmem_base + acc * acc_cols + (static_cast<uint32_t>(q * 32) << 16);
      // rows [lo, lo + nrows) of the tile's tile_m are this CTA's to sum
      const int rs = (pq.tile_m + S - 1) / S;
      const int lo = min(pq.tile_m, static_cast<int>(rank) * rs);
      const int nrows = min(pq.tile_m, lo + rs) - lo;
      if (S == 1) {
        // One split: the accumulator is the sum; store straight from registers.
        const int grow = t.m0 + row;
        for (int c = 0; c < pq.bn; c += 16) {
          uint32_t v[16];
          if (t.n_iter > 0) {
            tmem_ld16(t_base + static_cast<uint32_t>(c), v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = 0u;
          }
          if (grow >= pq.M || row >= pq.tile_m) continue;
          const int gcol = t.n0 + c;
          const int lim = min(pq.out_valid, pq.N);
          if (pq.red_f32_t) {
            // a warp's 32 rows are 32 consecutive outputs of each column
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (gcol + e < lim) {
                float* dst = pq.red_f32_t + static_cast<int64_t>(gcol + e + t.out_col0) * pq.red_ld_t + grow;
                *dst = red_out1(pq, dst, __fmul_rn(pq.red_scale, __uint_as_float(v[e])));
              }
          } else {
            const int64_t o = static_cast<int64_t>(grow) * pq.red_ld + t.out_col0 + gcol;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (gcol + 8 * h >= lim) continue;
              const float* f = reinterpret_cast<const float*>(v) + 8 * h;
              if (pq.red_bf16)
                *reinterpret_cast<uint4*>(pq.red_bf16 + o + 8 * h) =
                    make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                               pack_bf16x2(f[6], f[7]));
              if (pq.red_bf16_s) {
                float g8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) g8[e] = __fmul_rn(pq.red_scale, f[e]);
                *reinterpret_cast<uint4*>(pq.red_bf16_s + o + 8 * h) =
                    make_uint4(pack_bf16x2(g8[0], g8[1]), pack_bf16x2(g8[2], g8[3]), pack_bf16x2(g8[4], g8[5]),
                               pack_bf16x2(g8[6], g8[7]));
              }
              if (pq.red_f32) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  float* dst = pq.red_f32 + o + 8 * h + 4 * e;
                  *reinterpret_cast<float4*>(dst) = red_out4(
                      pq, dst,
                      make_float4(__fmul_rn(pq.red_scale, f[4 * e]), __fmul_rn(pq.red_scale, f[4 * e + 1]),
                                  __fmul_rn(pq.red_scale, f[4 * e + 2]), __fmul_rn(pq.red_scale, f[4 * e + 3])));
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        continue;
      }
      for (int c64 = 0; c64 < pq.bn; c64 += 64, ++round) {
        const int cw = min(64, pq.bn - c64);
        // 1. this CTA's buffer has been read by every CTA in the previous round
        if (!warp_wait_cluster(red_free, (round & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        // 2. accumulator columns [c64, c64 + cw) -> buffer row `row`
        for (int c = 0; c < cw; c += 16) {
          uint32_t v[16];
          if (t.n_iter > 0) {
            tmem_ld16(t_base + static_cast<uint32_t>(c64 + c), v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = 0u;
          }
          float4* dst = reinterpret_cast<float4*>(red + row * kRedLd + c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                 __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
        }
        if (c64 + 64 >= pq.bn) {  // accumulator read out: the MMA warp may reuse it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
        }
        // 3. publish: arrive (release) on every CTA's red_ready
        for (int k = 0; k < S; ++k) mbar_arrive_cluster(mapa_shared(ready_s, static_cast<uint32_t>(k)));
        // 4. every buffer of this round is written
        if (!warp_wait_cluster(red_ready, round & 1u, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        // 5. sum rows [lo, lo + nrows) over the cluster in split order; a
        //    thread takes groups of 4 columns, kB groups at a time so that
        //    kB loads are in flight per split.  Row-major outputs walk the
        //    groups row by row, the transposed output column-group by
        //    column-group (consecutive threads -> consecutive rows).
        constexpr int kB = 4;
        const int g4 = cw / 4;
        const int items = nrows * g4;
        const bool tr = pq.red_f32_t != nullptr;
        for (int base = et; base < items; base += 128 * kB) {
          uint32_t off[kB];
          int rr[kB], cc[kB];
          float4 sum[kB];
#pragma unroll
          for (int i = 0; i < kB; ++i) {
            const int e = min(base + 128 * i, items - 1);
            rr[i] = lo + (tr ? e % nrows : e / g4);
            cc[i] = 4 * (tr ? e / nrows : e % g4);
            off[i] = red_s + static_cast<uint32_t>(rr[i] * kRedLd + cc[i]) * 4u;
            sum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          for (int k = 0; k < S; ++k) {
            float4 v[kB];
#pragma unroll
            for (int i = 0; i < kB; ++i) v[i] = ld_shared_cluster_v4(mapa_shared(off[i], static_cast<uint32_t>(k)));
#pragma unroll
            for (int i = 0; i < kB; ++i) {
              sum[i].x += v[i].x;
              sum[i].y += v[i].y;
              sum[i].z += v[i].z;
              sum[i].w += v[i].w;
            }
          }
#pragma unroll
          for (int i = 0; i < kB; ++i) {
            if (base + 128 * i >= items) break;
            const int grow = t.m0 + rr[i], gcol = t.n0 + c64 + cc[i];
            if (grow >= pq.M || gcol >= pq.out_valid || gcol >= pq.N) continue;
            const float f[4] = {sum[i].x, sum[i].y, sum[i].z, sum[i].w};
            if (tr) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float* dst = pq.red_f32_t + static_cast<int64_t>(gcol + e + t.out_col0) * pq.red_ld_t + grow;
                *dst = red_out1(pq, dst, __fmul_rn(pq.red_scale, f[e]));
              }
              continue;
            }
            const int64_t o = static_cast<int64_t>(grow) * pq.red_ld + t.out_col0 + gcol;
            if (pq.red_bf16)
              *reinterpret_cast<uint2*>(pq.red_bf16 + o) = make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
            if (pq.red_bf16_s)
              *reinterpret_cast<uint2*>(pq.red_bf16_s + o) =
                  make_uint2(pack_bf16x2(__fmul_rn(pq.red_scale, f[0]), __fmul_rn(pq.red_scale, f[1])),
                             pack_bf16x2(__fmul_rn(pq.red_scale, f[2]), __fmul_rn(pq.red_scale, f[3])));
            if (pq.red_f32)
              *reinterpret_cast<float4*>(pq.red_f32 + o) =
                  red_out4(pq, pq.red_f32 + o,
                           make_float4(__fmul_rn(pq.red_scale, f[0]), __fmul_rn(pq.red_scale, f[1]),
                                       __fmul_rn(pq.red_scale, f[2]), __fmul_rn(pq.red_scale, f[3])));
          }
        }
        // 6. done reading this round: arrive (release) on every CTA's red_free
        for (int k = 0; k < S; ++k) mbar_arrive_cluster(mapa_shared(free_s, static_cast<uint32_t>(k)));
      }
    }
    if (!ok && lane == 0) {
      if (!*abort_flag) report(p, 32u);
      *abort_flag = 1;
    }
    if (p.dq_words > 0) dq_slice_warp(p, dq_ctr, lane);  // the rest of Wd, if any
    }  // if constexpr (RED)
  } else if (warp >= 2) {
    // ---------------- Epilogue ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    int j = 0;
    for (int T = walk_first; T < walk_total; T += walk_stride, ++j) {
      const TileInfo t = tile_info(p, T);
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
      const bool row_ok = grow < p.M && row < p.tile_m;
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
        if (EPI == EPI_F32_PART) {
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
  // No CTA leaves while a peer may still read its buffer or arrive on its
  // barriers (every wait above is bounded, so all threads get here).
  if (RED) cluster_sync_all();
}

}  // namespace qlora
