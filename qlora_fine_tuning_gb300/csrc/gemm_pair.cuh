// gemm_pair.cuh -- persistent tcgen05 GEMM on CTA pairs (.cta_group::2) for
// the two large contractions of the layer:
//   Y  = X . Wd^T + (s XA) . B       and      dX = dY . Wd + (s G) . A^T
// Both operands K-major, bf16 output.
//
// A cluster of two CTAs computes a 256 x 256 output tile with one
// tcgen05.mma.cta_group::2 (M=256, N=256, K=16) per 16-wide K step: each CTA
// holds 128 rows of A and 128 rows of B (half of N) in its own shared memory,
// and the accumulator rows of each CTA live in its own TMEM.  Compared with a
// single-CTA 128 x 256 tile this halves the B bytes each SM stages and feeds
// to the tensor core per K step, which is what bounds the single-CTA kernel.
//
// Roles per CTA (6 warps; issuing roles run as whole warps and one elected
// lane issues, keeping every operand warp-uniform):
//   warp 0         TMA producer for this CTA's halves; completion is counted
//                  on the even CTA's "full" barrier (it expects both halves);
//   warp 1         (even CTA only) MMA issuer; commits multicast to both
//                  CTAs' "empty" / "accumulator full" barriers;
//   warps 2..5     epilogue for this CTA's 128 rows; release the accumulator
//                  by arriving on the even CTA's "accumulator empty" barrier.
// Two TMEM accumulators of 256 columns (512 columns, allocated for the pair).
//
// FUSED_DQ: the B operand is the frozen 4-bit weight itself.  Per stage the
// producer brings this CTA's packed codes and absmax in by TMA into a staging
// area; 8 more warps (6..13) expand them -- fp32 product codebook * absmax,
// round-to-nearest-even to bf16, exactly as dequant_4bit -- straight into the
// 128-byte-swizzled B tile (K-major for Y, MN-major for dX), make the writes
// visible to the tensor core (fence.proxy.async) and arrive on the even CTA's
// "full" barrier next to the TMA bytes of A.  No dequantised copy of W is
// ever written to memory.
//
// Measured on GB300 this variant is ~3x slower than dequantising W once per
// call with dequant4_kernel and feeding bf16 tiles by TMA: the expansion adds
// several hand-offs (staging TMA, dequant-warp wake-up, proxy fence,
// cross-CTA arrival) to every stage's turnaround, which the 5-stage ring
// (38 KiB stages) cannot hide.  The library therefore runs it only on request
// (QLORA_FUSED_DQ=1).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace qlora {

constexpr uint32_t kPairStageBytes = 2 * 128 * 128;  // A half + B half, 64-wide K block
constexpr uint32_t kRawBytes = 4096 + 2048;           // packed codes + absmax box
constexpr uint32_t kPairDqStageBytes = 38912;         // A + B + raw, rounded to 1 KiB
constexpr int kDqWarps = 8;

// One dequant thread expands 32 codes (16 packed bytes) of one smem row into
// four swizzled 16-byte chunks of bf16: chunk `c0 + c` of row `row` of the
// 64-wide block at `blk`.
__device__ __forceinline__ void dq_row32(const uint8_t* packed16, float am, const float* cb, uint8_t* blk, int row,
                                         int c0) {
  const uint4 pk = *reinterpret_cast<const uint4*>(packed16);
  const uint32_t words[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t o[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t byte = (words[c] >> (8 * b)) & 0xFFu;
      o[b] = pack_bf16x2(__fmul_rn(cb[byte & 0xFu], am), __fmul_rn(cb[byte >> 4], am));
    }
    const int chunk = (c0 + c) ^ (row & 7);
    *reinterpret_cast<uint4*>(blk + row * 128 + chunk * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Tile order.  group_m > 0: bands of group_m row tiles, the row tile running
// fastest within a band, then the column tile.  group_m < 0: bands of
// -group_m column tiles, the column tile running fastest, then the row tile.
// Tiles processed at the same time then share one band of an operand, which
// stays in L2 while the other operand streams past it once per band.
__device__ __forceinline__ void pair_tile_coords(const GemmArgs& p, int tile, int& mt, int& nt) {
  if (p.group_m < 0 && -p.group_m < p.n_tiles) {
    const int gn = -p.group_m;
    const int band_tiles = gn * p.m_tiles;
    const int band = tile / band_tiles;
    const int in_band = tile - band * band_tiles;
    const int cols = min(gn, p.n_tiles - band * gn);  // the last band may be narrower
    nt = band * gn + in_band % cols;
    mt = in_band / cols;
    return;
  }
  const int gm = (p.group_m > 0 && p.group_m < p.m_tiles) ? p.group_m : p.m_tiles;
  const int band_tiles = gm * p.n_tiles;
  const int band = tile / band_tiles;
  const int in_band = tile - band * band_tiles;
  const int rows = min(gm, p.m_tiles - band * gm);
  mt = band * gm + in_band % rows;
  nt = in_band / rows;
}

// B_MN: B is read MN-major (its rows are reduction rows holding 64 output
// columns each; used for dX straight from the row-major dequantised weight).
// The rank-r steps read B2 the other way round: MN-major in the forward
// (B [r,N] as stored), K-major for dX (A [K,R] as stored).
// With FUSED_DQ, tmB maps the packed codes (uint8 [N, K/2]) and tmS the
// absmax (fp32 [N, K/64]); otherwise tmB maps the bf16 B operand and tmS is
// unused.
template <bool B_MN, bool FUSED_DQ>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FUSED_DQ ? 448 : 192, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                     const __grid_constant__ CUtensorMap tmS, const GemmArgs p) {
  constexpr uint32_t kStage = FUSED_DQ ? kPairDqStageBytes : kPairStageBytes;
  // The rank-r B-operand is read MN-major exactly when the main one is not:
  // forward B2 = B [r,N] (rows = rank index), dX B2 = A [K,R] (rows = output).
  constexpr bool B2_MN = !B_MN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((((raw + 1023u) & ~1023u)) - raw);
  uint8_t* ctrl = smem + static_cast<uint32_t>(p.stages) * kStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint64_t* raw_full = mma_done + 1;  // [kMaxStages] packed codes + absmax landed (FUSED_DQ)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(raw_full + kMaxStages);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);
  float* cb_s = reinterpret_cast<float*>(tmem_slot + 4);  // [16] codebook (FUSED_DQ)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int npairs = static_cast<int>(gridDim.x >> 1);
  const int total = p.m_tiles * p.n_tiles;
  const bool has_lora = p.lora_atoms > 0;
  const int nkb = (p.red_len + 63) / 64;
  constexpr uint32_t kAccCols = 256;
  constexpr uint32_t kTmemCols = 512;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages; ++i) {
      // TMA arrival of the even CTA, plus every dequant warp of both CTAs
      mbar_init(&full[i], FUSED_DQ ? 1 + 2 * kDqWarps : 1);
      mbar_init(&empty[i], 1);
      mbar_init(&raw_full[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 8);  // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
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
  cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();  // the predecessor kernel's global writes are visible from here on
  griddep_launch_dependents();
  if (FUSED_DQ && threadIdx.x < 16) cb_s[threadIdx.x] = p.codebook[threadIdx.x];
  if (FUSED_DQ) __syncthreads();
  const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);      // even CTA's ring barriers
  const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);  // even CTA's accumulator-empty

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs; whole warp, elected lane issues) ----------------
    const uint32_t tx_pair = 2u * kPairStageBytes;
    const uint32_t tx_a_pair = 2u * kATileBytes;
    const uint32_t tx_raw = B_MN ? 4096u + 1024u : 4096u + 2048u;
    // The operand of the current band is re-read by the band's tiles: keep it
    // (evict-last); the other operand streams past once per band (evict-first).
    // Row bands hold rows of A, column bands (group_m < 0) columns of B.
    const bool band_is_b = p.group_m < 0 && -p.group_m < p.n_tiles;
    const uint64_t keep = (p.l2_hints & 2) ? l2_policy_evict_last() : l2_policy_evict_normal();
    const uint64_t pass = (p.l2_hints & 4) ? l2_policy_evict_first() : l2_policy_evict_normal();
    const uint64_t pol_a = band_is_b ? pass : keep;
    const uint64_t pol_b = band_is_b ? keep : pass;
    uint32_t g = 0;
    uint32_t raw_issued = 0;  // bit i: ring position g-1-i had a packed-code load in flight
    bool ok = true;
    for (int tile = pair; tile < total && ok; tile += npairs) {
      int mt, nt;
      pair_tile_coords(p, tile, mt, nt);
      const int m0 = mt * 256 + static_cast<int>(rank) * 128;  // this CTA's rows of A / output
      const int nb = nt * 256;
      const int n0 = nb + static_cast<int>(rank) * 128;        // this CTA's rows of B
      const int sg = (p.mode == GM_FWD) ? seg_index(p, nb) : 0;
      const int a2_x0 = (p.mode == GM_FWD) ? sg * p.r : 0;
      const int n_iter = nkb + (has_lora ? p.lora_atoms : 0);
      for (int it = 0; it < n_iter; ++it) {
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
        raw_issued <<= 1;
        // Test hook: the even CTA of pair 0 never arms stage 0's "full"
        // barrier, so the MMA wait on it runs out.  (With FUSED_DQ the packed
        // codes still come in below: the dequant warps stay in step with the
        // ring and never arrive twice in one phase.)
        const bool stall = p.debug_stall && g == 0 && pair == 0 && rank == 0;
        if (stall && !FUSED_DQ) {
          ++g;
          continue;
        }
        uint8_t* a_dst = smem + s * kStage;
        uint8_t* b_dst = a_dst + kATileBytes;
        const uint32_t bar = full0 + s * 8u;
        if (FUSED_DQ && it < nkb) {
          // A by TMA; B arrives as packed codes + absmax and is expanded in smem
          const int kel = it * 64;
          uint8_t* r_dst = b_dst + kATileBytes;
          if (!stall) {
            if (rank == 0) mbar_arrive_expect_tx_ws(&full[s], tx_a_pair);
            tma_load_2d_pair_hint_ws(a_dst, &tmA, bar, kel, m0, pol_a);
          }
          mbar_arrive_expect_tx_ws(&raw_full[s], tx_raw);
          if (B_MN) {
            // rows = reduction index n (64 of them), 128 output columns k
            tma_load_2d_ws(r_dst, &tmB, &raw_full[s], n0 / 2, kel);
            tma_load_2d_ws(r_dst + 4096, &tmS, &raw_full[s], (n0 / 64) & ~3, kel);
          } else {
            // rows = output index n (128 of them), 64 reduction columns k
            tma_load_2d_ws(r_dst, &tmB, &raw_full[s], kel / 2, n0);
            tma_load_2d_ws(r_dst + 4096, &tmS, &raw_full[s], it & ~3, n0);
          }
          raw_issued |= 1u;
          ++g;
          continue;
        }
        if (FUSED_DQ) {
          // rank-r step: nothing to expand, but the staging barrier still
          // completes one phase per ring round so its parity tracks `g`
          if (lane == 0) mbar_arrive(&raw_full[s]);
          __syncwarp();
        }
        if (rank == 0) mbar_arrive_expect_tx_ws(&full[s], tx_pair);
        if (it < nkb) {
          const int kel = it * 64;
          tma_load_2d_pair_hint_ws(a_dst, &tmA, bar, kel, m0, pol_a);
          if (B_MN) {
            tma_load_2d_pair_hint_ws(b_dst, &tmB, bar, n0, kel, pol_b);
            tma_load_2d_pair_hint_ws(b_dst + 8192, &tmB, bar, n0 + 64, kel, pol_b);
          } else {
            tma_load_2d_pair_hint_ws(b_dst, &tmB, bar, kel, n0, pol_b);
          }
        } else {
          const int a = it - nkb;
          tma_load_2d_pair_ws(a_dst, &tmA2, bar, a2_x0 + 64 * a, m0);
          if (B2_MN) {
            tma_load_2d_pair_ws(b_dst, &tmB2, bar, n0, 64 * a);
            tma_load_2d_pair_ws(b_dst + 8192, &tmB2, bar, n0 + 64, 64 * a);
          } else {
            tma_load_2d_pair_ws(b_dst, &tmB2, bar, 64 * a, n0);
          }
        }
        ++g;
      }
    }
    if (lane == 0) {
      const uint32_t S = static_cast<uint32_t>(p.stages);
      for (uint32_t q = (g > S ? g - S : 0u); q < g; ++q) {
        if (rank == 0) mbar_wait(&full[q % S], (q / S) & 1u, p.timeout_ns);
        if (FUSED_DQ && ((raw_issued >> (g - 1 - q)) & 1u)) mbar_wait(&raw_full[q % S], (q / S) & 1u, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (even CTA; whole warp, elected lane issues) ----------------
    if (rank == 0) {
      const uint32_t idesc = idesc_bf16_f32(256, 256, false, B_MN);
      const uint32_t idesc_lora = idesc_bf16_f32(256, 256, false, B2_MN);
      uint32_t g = 0;
      int j = 0;
      bool ok = true;
      for (int tile = pair; tile < total && ok; tile += npairs, ++j) {
        const uint32_t acc = static_cast<uint32_t>(j & 1);
        if (!warp_wait(&tempty[acc], (static_cast<uint32_t>(j >> 1) & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
          if (lane == 0) {
            if (!*abort_flag) report(p, 8u);
            *abort_flag = 1;
          }
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kAccCols;
        const int n_iter = nkb + (has_lora ? p.lora_atoms : 0);
        for (int it = 0; it < n_iter; ++it) {
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
          const uint32_t a_addr = smem_u32(smem + s * kStage);
          const uint32_t b_addr = a_addr + kATileBytes;
          if (it < nkb) {
            const uint64_t bd = B_MN ? sdesc_sw128(b_addr, 8192u, 1024u) : sdesc_sw128(b_addr, 16u, 1024u);
            tc_mma_bf16_pair_k64_ws(d_tmem, sdesc_sw128(a_addr, 16u, 1024u), bd, 2u, B_MN ? (2048u >> 4) : 2u,
                                    idesc, it > 0 ? 1u : 0u);
          } else {
            const int ksteps = min(4, p.lora_ksteps - 4 * (it - nkb));
            for (int kk = 0; kk < ksteps; ++kk)
              tc_mma_bf16_pair_ws(d_tmem, sdesc_sw128(a_addr + static_cast<uint32_t>(kk) * 32u, 16u, 1024u),
                                  B2_MN ? sdesc_sw128(b_addr + static_cast<uint32_t>(kk) * 2048u, 8192u, 1024u)
                                        : sdesc_sw128(b_addr + static_cast<uint32_t>(kk) * 32u, 16u, 1024u),
                                  idesc_lora, (it > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit_pair_multicast_ws(&empty[s], 0x3);
          ++g;
        }
        if (!ok) break;
        tc_commit_pair_multicast_ws(&tfull[acc], 0x3);
      }
      tc_commit_pair_multicast_ws(mma_done, 0x3);
    }
  } else if (warp >= 2 && warp < 6) {
    // ---------------- Epilogue (both CTAs, own 128 rows) ----------------
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int j = 0;
    for (int tile = pair; tile < total; tile += npairs, ++j) {
      int mt, nt;
      pair_tile_coords(p, tile, mt, nt);
      const uint32_t acc = static_cast<uint32_t>(j & 1);
      if (!warp_wait(&tfull[acc], static_cast<uint32_t>(j >> 1) & 1u, p.timeout_ns, abort_flag)) {
        if (lane == 0) {
          if (!*abort_flag) report(p, 4u);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const int grow = mt * 256 + static_cast<int>(rank) * 128 + row;
      const bool row_ok = grow < p.M;
      const uint32_t t_base = tmem_base + acc * kAccCols + (static_cast<uint32_t>(q * 32) << 16);
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(grow) * p.out_ld;
      for (int c = 0; c < 16; ++c) {
        uint32_t v[16];
        tmem_ld16(t_base + static_cast<uint32_t>(c * 16), v);
        tmem_ld_wait();
        if (!row_ok) continue;
        const int c0 = nt * 256 + c * 16;
#pragma unroll
        for (int gq = 0; gq < 2; ++gq) {
          const int col = c0 + gq * 8;
          if (col < p.N) {
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(&tempty[acc]);
        else mbar_arrive_cluster(tempty0 + acc * 8u);
      }
    }
  }
  else if (FUSED_DQ && warp >= 6) {
    // ---------------- In-kernel dequantisation (both CTAs, this CTA's half of B) ----------------
    const int t = threadIdx.x - 6 * 32;  // 0..255
    const uint32_t full_s0 = full0;      // even CTA's full barriers (cluster address)
    uint32_t g = 0;
    bool ok = true;
    for (int tile = pair; tile < total && ok; tile += npairs) {
      int mt, nt;
      pair_tile_coords(p, tile, mt, nt);
      const int n0 = nt * 256 + static_cast<int>(rank) * 128;
      const int n_iter = nkb + (has_lora ? p.lora_atoms : 0);
      for (int it = 0; it < n_iter; ++it) {
        const uint32_t s = g % static_cast<uint32_t>(p.stages);
        const uint32_t ph = (g / static_cast<uint32_t>(p.stages)) & 1u;
        // one staging phase per ring round (rank-r rounds complete it with a plain arrive)
        if (!warp_wait(&raw_full[s], ph, p.timeout_ns, abort_flag)) {
          if (lane == 0) {
            if (!*abort_flag) report(p, 16u);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
        if (it < nkb) {
          uint8_t* b_blk = smem + s * kStage + kATileBytes;
          const uint8_t* rw = b_blk + kATileBytes;
          const float* am_box = reinterpret_cast<const float*>(rw + 4096);
          if (B_MN) {
            // 64 reduction rows x 128 output columns: thread -> row t/4, 32 columns
            const int row = t >> 2, q4 = t & 3, h = q4 >> 1;
            const float am = am_box[row * 4 + ((n0 >> 6) & 3) + h];
            dq_row32(rw + row * 64 + q4 * 16, am, cb_s, b_blk + h * 8192, row, (q4 & 1) * 4);
          } else {
            // 128 output rows x 64 reduction columns: thread -> row t/2, 32 columns
            const int row = t >> 1, hh = t & 1;
            const float am = am_box[row * 4 + (it & 3)];
            dq_row32(rw + row * 32 + hh * 16, am, cb_s, b_blk, row, hh * 4);
          }
          fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
        }
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(&full[s]);
          else mbar_arrive_cluster(full_s0 + s * 8u);
        }
        ++g;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0) mbar_wait(mma_done, 0u, p.timeout_ns);  // no MMA still writes our TMEM
  __syncwarp();
  cluster_sync_all();  // the peer is done with the pair's TMEM too
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace qlora
