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
// FUSED_DQ: the B operand is the frozen 4-bit weight itself, expanded inside
// the kernel; no dequantised copy of W is ever written to memory.  Eight more
// warps (6..13) per CTA own this CTA's half of every B tile: each thread
// copies its 16 bytes of packed codes (32 weights) and their absmax by
// cp.async into a small ring of its own, kDqAhead ring positions ahead of use.
// Once the MMAs have released the stage, it builds the 16 possible values of
// its block -- bf16( fp32( codebook[i] * absmax ) ), the same fp32 product and
// round-to-nearest-even as dequant_4bit -- as two byte planes in registers,
// turns every nibble into its value with byte permutes (no per-weight
// shared-memory lookup), writes the 128-byte-swizzled B tile (K-major for Y,
// MN-major for dX), makes the writes visible to the tensor core
// (fence.proxy.async) and arrives on the even CTA's "full" barrier next to the
// TMA bytes of A.
//
// Measured on GB300 this variant is ~1.8x slower than dequantising W once per
// call (dequant_4bit) and feeding bf16 tiles by TMA: with the expansion taken
// out entirely (raw copies written instead) the hand-off through generic
// shared-memory writes alone costs ~30%, and the expansion -- each weight is
// expanded once per 256-row tile that uses it -- the rest: its permutes,
// logic ops and shifts run on the half-rate integer pipe, ~670 cycles of it
// per CTA and stage against ~512 cycles for the stage's MMAs.  The library
// runs it only on request (QLORA_FUSED_DQ=1).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace qlora {

constexpr uint32_t kPairStageBytes = 2 * 128 * 128;  // A half + B half, 64-wide K block
constexpr int kDqWarps = 8;                           // in-kernel dequantisation warps per CTA
constexpr int kDqAhead = 4;                           // ring positions a code copy runs ahead
constexpr int kDqSlots = kDqAhead + 1;                // code slots (one is being read)
constexpr uint32_t kDqSlotBytes = 32 * kDqWarps * (16 + 4);  // 16 B of codes + 4 B absmax per thread

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// The 16 values one 64-block can take, T[i] = bf16(fp32(cb[i] * am)), as two
// byte planes: lo[q] holds the low bytes of T[4q..4q+3], hi[q] the high bytes.
// cb2[j] holds codebook entries 2j and 2j+1; each paired multiply rounds both
// products to nearest like two single ones.
__device__ __forceinline__ void dq_table(const uint64_t (&cb2)[8], float am, uint32_t (&lo)[4], uint32_t (&hi)[4]) {
  uint64_t am2;
  asm("mov.b64 %0, {%1, %1};" : "=l"(am2) : "f"(am));
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint64_t p0, p1;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p0) : "l"(cb2[2 * q]), "l"(am2));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p1) : "l"(cb2[2 * q + 1]), "l"(am2));
    float f0, f1, f2, f3;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f0), "=f"(f1) : "l"(p0));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f2), "=f"(f3) : "l"(p1));
    const uint32_t a = pack_bf16x2(f0, f1);
    const uint32_t b = pack_bf16x2(f2, f3);
    lo[q] = prmt(a, b, 0x6420u);
    hi[q] = prmt(a, b, 0x7531u);
  }
}

// Eight codes (one 32-bit word, code j in nibble j) -> eight bf16 values in
// order.  A permute picks bytes from an 8-byte pair of planes by the low three
// bits of each code (entries 0-7 and 8-15 separately); a third permute keeps,
// per byte, the half that bit 3 of the code selects; two more interleave the
// low and high bytes into bf16 pairs.
__device__ __forceinline__ uint4 dq_word(uint32_t w, const uint32_t (&lo)[4], const uint32_t (&hi)[4]) {
  const uint32_t s1 = w & 0x77777777u;
  const uint32_t s2 = ((w >> 1) & 0x44444444u) | 0x32103210u;
  uint4 o;
  {
    const uint32_t l = prmt(prmt(lo[0], lo[1], s1), prmt(lo[2], lo[3], s1), s2);
    const uint32_t h = prmt(prmt(hi[0], hi[1], s1), prmt(hi[2], hi[3], s1), s2);
    o.x = prmt(l, h, 0x5140u);
    o.y = prmt(l, h, 0x7362u);
  }
  {
    const uint32_t u1 = s1 >> 16, u2 = s2 >> 16;
    const uint32_t l = prmt(prmt(lo[0], lo[1], u1), prmt(lo[2], lo[3], u1), u2);
    const uint32_t h = prmt(prmt(hi[0], hi[1], u1), prmt(hi[2], hi[3], u1), u2);
    o.z = prmt(l, h, 0x5140u);
    o.w = prmt(l, h, 0x7362u);
  }
  return o;
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
// columns each; used for dX straight from the row-major weight).
// The rank-r steps read B2 the other way round: MN-major in the forward
// (B [r,N] as stored), K-major for dX (A [K,R] as stored).
// Without FUSED_DQ tmB maps the bf16 dequantised weight; with it tmB is unused
// and the dequantisation warps read p.dq_idx / p.dq_absmax directly.
template <bool B_MN, bool FUSED_DQ>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FUSED_DQ ? 192 + 32 * kDqWarps : 192, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                     const GemmArgs p) {
  constexpr uint32_t kStage = kPairStageBytes;
  // The rank-r B-operand is read MN-major exactly when the main one is not:
  // forward B2 = B [r,N] (rows = rank index), dX B2 = A [K,R] (rows = output).
  constexpr bool B2_MN = !B_MN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((((raw + 1023u) & ~1023u)) - raw);
  // FUSED_DQ: the code slots of the dequantisation warps follow the ring
  uint8_t* cring = smem + static_cast<uint32_t>(p.stages) * kStage;
  uint8_t* ctrl = cring + (FUSED_DQ ? kDqSlots * kDqSlotBytes : 0u);
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

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
      // TMA arrival of the even CTA, plus every dequantisation warp of both CTAs
      mbar_init(&full[i], FUSED_DQ ? 1 + 2 * kDqWarps : 1);
      mbar_init(&empty[i], 1);
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
    if (!FUSED_DQ) tma_prefetch_desc(&tmB);
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
  const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);      // even CTA's ring barriers
  const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);  // even CTA's accumulator-empty

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs; whole warp, elected lane issues) ----------------
    const uint32_t tx_pair = 2u * kPairStageBytes;
    const uint32_t tx_a_pair = 2u * kATileBytes;
    // The operand of the current band is re-read by the band's tiles: keep it
    // (evict-last); the other operand streams past once per band (evict-first).
    // Row bands hold rows of A, column bands (group_m < 0) columns of B.
    const bool band_is_b = p.group_m < 0 && -p.group_m < p.n_tiles;
    const uint64_t keep = (p.l2_hints & 2) ? l2_policy_evict_last() : l2_policy_evict_normal();
    const uint64_t pass = (p.l2_hints & 4) ? l2_policy_evict_first() : l2_policy_evict_normal();
    const uint64_t pol_a = band_is_b ? pass : keep;
    const uint64_t pol_b = band_is_b ? keep : pass;
    uint32_t g = 0;
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
        // Test hook: the even CTA of pair 0 never arms stage 0's "full"
        // barrier, so the MMA wait on it runs out.
        if (p.debug_stall && g == 0 && pair == 0 && rank == 0) {
          ++g;
          continue;
        }
        uint8_t* a_dst = smem + s * kStage;
        uint8_t* b_dst = a_dst + kATileBytes;
        const uint32_t bar = full0 + s * 8u;
        if (it < nkb) {
          const int kel = it * 64;
          if (rank == 0) mbar_arrive_expect_tx_ws(&full[s], FUSED_DQ ? tx_a_pair : tx_pair);
          tma_load_2d_pair_hint_ws(a_dst, &tmA, bar, kel, m0, pol_a);
          if (!FUSED_DQ) {  // else the dequantisation warps write the B half
            if (B_MN) {
              tma_load_2d_pair_hint_ws(b_dst, &tmB, bar, n0, kel, pol_b);
              tma_load_2d_pair_hint_ws(b_dst + 8192, &tmB, bar, n0 + 64, kel, pol_b);
            } else {
              tma_load_2d_pair_hint_ws(b_dst, &tmB, bar, kel, n0, pol_b);
            }
          }
        } else {
          const int a = it - nkb;
          if (rank == 0) mbar_arrive_expect_tx_ws(&full[s], tx_pair);
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
    if (lane == 0 && rank == 0) {
      // do not leave while copies this pair issued may still land in smem
      const uint32_t S = static_cast<uint32_t>(p.stages);
      for (uint32_t q = (g > S ? g - S : 0u); q < g; ++q) mbar_wait(&full[q % S], (q / S) & 1u, p.timeout_ns);
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
      if (!warp_wait_sleepy(&tfull[acc], static_cast<uint32_t>(j >> 1) & 1u, p.timeout_ns, abort_flag)) {
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
  } else if constexpr (FUSED_DQ) {
    // ---------------- In-kernel dequantisation (both CTAs, this CTA's half of B) ----------------
    // Thread t owns 32 consecutive weights of one 64-block per stage, always
    // at the same place in the B tile:
    //   Y  (B K-major, 128 output rows n x 64 reduction k): row t/2, k half t%2;
    //   dX (B MN-major, 64 reduction rows n x 128 output cols k): row t/4,
    //      32 columns (t%4)*32.. (the 64-column block (t%4)/2).
    // Its 16 bytes of codes and its absmax come in by cp.async, kDqAhead ring
    // positions ahead, into its own place in a slot of `cring` (asynchronous
    // copies: the release of the arrival on "full" below does not wait for
    // them).
    const int t = static_cast<int>(threadIdx.x) - 192;  // 0..255
    const int n_w = B_MN ? p.red_len : p.N;             // rows of the 4-bit weight
    const int k_w = p.dq_k;                             // its columns
    const int64_t row_bytes = k_w / 2;                  // packed codes per weight row
    const int blocks_per_row = k_w / 64;
    const int trow = B_MN ? (t >> 2) : (t >> 1);
    const int tq = B_MN ? (t & 3) : (t & 1);
    uint32_t off[4];  // this thread's four 16-byte chunks inside a stage's B half
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int chunk = (B_MN ? (tq & 1) * 4 : tq * 4) + c;
      off[c] = static_cast<uint32_t>((B_MN ? (tq >> 1) * 8192 : 0) + trow * 128 + ((chunk ^ (trow & 7)) * 16));
    }
    uint64_t cb2[8];
    {
      const ulonglong2* c4 = reinterpret_cast<const ulonglong2*>(p.codebook);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const ulonglong2 v = __ldg(c4 + i);
        cb2[2 * i] = v.x;
        cb2[2 * i + 1] = v.y;
      }
    }
    const uint32_t my_codes = smem_u32(cring) + static_cast<uint32_t>(t) * 16u;
    const uint32_t my_am = smem_u32(cring) + 4096u + static_cast<uint32_t>(t) * 4u;
    const uint32_t b_base = smem_u32(smem) + kATileBytes;
    const int n_iter = nkb + (has_lora ? p.lora_atoms : 0);
    const int my_tiles = pair < total ? (total - pair + npairs - 1) / npairs : 0;
    // Copy walker: tile jt_a, k-block it_a; the source of the next copy and
    // its step per k-block.
    int jt_a = 0, it_a = 0, n_a = 0;
    bool tile_ok = false;
    const uint8_t* src_c = nullptr;
    const float* src_a = nullptr;
    const int64_t step_c = B_MN ? 64 * row_bytes : 32;
    const int64_t step_a = B_MN ? int64_t(64) * blocks_per_row : 1;
    auto start_tile = [&](int jt) {
      int mt, nt;
      pair_tile_coords(p, pair + jt * npairs, mt, nt);
      const int c0 = nt * 256 + static_cast<int>(rank) * 128;  // this CTA's first B row (Y) / column (dX)
      const int n = B_MN ? trow : c0 + trow;
      const int k = B_MN ? c0 + tq * 32 : tq * 32;
      tile_ok = B_MN ? (k < k_w) : (n < n_w);
      n_a = n;
      src_c = p.dq_idx + static_cast<int64_t>(n) * row_bytes + k / 2;
      src_a = p.dq_absmax + static_cast<int64_t>(n) * blocks_per_row + k / 64;
    };
    if (my_tiles > 0) start_tile(0);
    uint32_t so_a = 0;   // byte offset of the slot the next copy goes to
    uint32_t vmask = 0;  // bit j: slot j holds codes from inside the weight
    uint32_t slot_a = 0;
    auto copy_next = [&]() {
      const bool v = jt_a < my_tiles && it_a < nkb && tile_ok && n_a < n_w;
      if (v) {
        cp_async_16(my_codes + so_a, src_c);
        cp_async_4(my_am + so_a, src_a);
      }
      cp_async_commit();  // one group per position, empty ones included
      vmask = (vmask & ~(1u << slot_a)) | (static_cast<uint32_t>(v) << slot_a);
      if (++slot_a == kDqSlots) {
        slot_a = 0;
        so_a = 0;
      } else {
        so_a += kDqSlotBytes;
      }
      if (jt_a < my_tiles) {
        src_c += step_c;
        src_a += step_a;
        if (B_MN) n_a += 64;
        if (++it_a == n_iter) {
          it_a = 0;
          if (++jt_a < my_tiles) start_tile(jt_a);
        }
      }
    };
#pragma unroll
    for (int q = 0; q < kDqAhead; ++q) copy_next();
    uint32_t s = 0, ph = 0, slot = 0, so = 0;
    bool ok = true;
    for (int jt = 0; jt < my_tiles && ok; ++jt) {
      for (int it = 0; it < n_iter; ++it) {
        // the MMAs that read this stage last round have completed
        if (!warp_wait(&empty[s], ph ^ 1u, p.timeout_ns, abort_flag)) {
          if (lane == 0) {
            if (!*abort_flag) report(p, 16u);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
        if (it < nkb) {
          const uint32_t b_s = b_base + s * kStage;
          cp_async_wait<kDqAhead - 1>();  // this position's copies have landed
          if ((vmask >> slot) & 1u) {
            uint4 cw;
            float am;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(cw.x), "=r"(cw.y), "=r"(cw.z), "=r"(cw.w)
                         : "r"(my_codes + so));
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(am) : "r"(my_am + so));
            uint32_t lo[4], hi[4];
            dq_table(cb2, am, lo, hi);
            const uint4 o0 = dq_word(cw.x, lo, hi), o1 = dq_word(cw.y, lo, hi);
            const uint4 o2 = dq_word(cw.z, lo, hi), o3 = dq_word(cw.w, lo, hi);
            st_shared_v4(b_s + off[0], o0);
            st_shared_v4(b_s + off[1], o1);
            st_shared_v4(b_s + off[2], o2);
            st_shared_v4(b_s + off[3], o3);
          } else {  // rows past the weight (reduction rows for dX must be zero)
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int c = 0; c < 4; ++c) st_shared_v4(b_s + off[c], z);
          }
          fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
        }
        copy_next();  // into the slot read one position ago
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(&full[s]);
          else mbar_arrive_remote_cta(full0 + s * 8u);
        }
        if (++s == static_cast<uint32_t>(p.stages)) {
          s = 0;
          ph ^= 1u;
        }
        if (++slot == kDqSlots) {
          slot = 0;
          so = 0;
        } else {
          so += kDqSlotBytes;
        }
      }
    }
    cp_async_wait<0>();  // no copy into this CTA's shared memory still in flight
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
