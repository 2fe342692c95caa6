// qlora_api.cu -- host side of libqlora.so: argument checks, workspace
// carving, TMA descriptor encoding, launch sequencing, profiler.
//
// Forward (one call, 3 launches):
//   dequant W -> Wd bf16 [N,K]            (elementwise, HBM-bound)
//   XA = X . A        rank-r GEMM, A read MN-major as stored; the splits of K
//                     are summed on chip -> XA_save and s*XA (bf16)
//   Y  = X . Wd^T + (s*XA) . B   CTA-pair GEMM, the rank-r product as extra
//                                 K-steps into the same TMEM accumulator
//                                 (B read MN-major as stored)
// Backward (one call, 4 launches):
//   G  = dY . B^T per segment     rank-r GEMM, splits of N summed on chip
//                                 -> s*G and G [M,R]
//   dequant W -> Wd bf16 [N,K]    (read MN-major by the dX GEMM)
//   dX = dY . Wd + (s*G) . A^T    CTA-pair GEMM, rank-r product as extra K-steps
//   dA = s X^T G and dB = s XA^T dY   one rank-r launch with two problems,
//                                 every operand read MN-major as stored
// When adapter boundaries are not multiples of 256 columns (or pairs are
// disabled) the products run on the single-CTA GEMM instead, with B^T and the
// transposed dequantisation it needs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/qlora.h"
#include "elementwise.cuh"
#include "gemm_pair.cuh"
#include "gemm_tc.cuh"

using namespace qlora;

namespace {

// ---------------------------------------------------------------------------
// Settings, profiler
// ---------------------------------------------------------------------------
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

// Test hook: label of the next GEMM launch that must stall (empty = none).
std::mutex g_stall_mu;
char g_stall_label[32] = {0};

bool take_stall(const char* name) {
  std::lock_guard<std::mutex> lk(g_stall_mu);
  if (g_stall_label[0] == 0 || std::strcmp(g_stall_label, name) != 0) return false;
  g_stall_label[0] = 0;
  return true;
}
std::atomic<uint64_t> g_launches{0};

struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pool_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Bracket one launch with events when the profiler is on.
struct LaunchScope {
  const char* name;
  cudaStream_t st;
  cudaEvent_t a = nullptr, b = nullptr;
  LaunchScope(const char* n, cudaStream_t s) : name(n), st(s) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof_on) {
      a = pool_event();
      b = pool_event();
      cudaEventRecord(a, st);
    }
  }
  ~LaunchScope() {
    if (a) {
      cudaEventRecord(b, st);
      std::lock_guard<std::mutex> lk(g_prof_mu);
      g_prof_recs.push_back({name, a, b});
    }
  }
};

// ---------------------------------------------------------------------------
// TMA descriptors (driver entry point fetched through the runtime, so the
// library does not link libcuda directly)
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor [outer, inner] with row stride ld (elements), box
// {64, box_outer}, 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t ld, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Shapes, workspace
// ---------------------------------------------------------------------------
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t rup(int64_t a, int64_t b) { return cdiv(a, b) * b; }
constexpr int kSMs = 152;

// Number of SMs of device `dev` (cached; 152 on GB300).
int cur_dev() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}

int sm_count(int dev) {
  static std::atomic<int> cache[64];
  int v = cache[dev & 63].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = kSMs;
  cache[dev & 63].store(v, std::memory_order_relaxed);
  return v;
}
constexpr int kMaxSplits = 8;

// Split count that depends only on the reduction length, so that a row's
// result never depends on how many rows are in the batch.
// Workspace header: the device error word (first 4 bytes of 256).
constexpr size_t kHeaderBytes = 256;

struct Layout {
  int64_t M, N, K, r, nseg, R, Rp, Mp;
  size_t off_err, off_wd, off_bt, off_xas, off_g, total;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

Layout layout(int64_t M, int64_t N, int64_t K, int64_t r, int64_t nseg) {
  Layout L{};
  L.M = M;
  L.N = N;
  L.K = K;
  L.r = r;
  L.nseg = nseg;
  L.R = r * nseg;
  L.Rp = rup(r, 16);
  L.Mp = rup(std::max<int64_t>(M, 1), 8);
  const size_t rows = size_t(std::max<int64_t>(M, 1));
  size_t o = 0;
  L.off_err = o;
  o += kHeaderBytes;
  L.off_wd = o;  // deq(W) [N,K] bf16
  o = align256(o + size_t(N) * K * 2);
  L.off_bt = o;  // B^T [N,Rp] bf16, zero columns r..Rp-1 (forward)
  o = align256(o + size_t(N) * L.Rp * 2);
  L.off_xas = o;  // s*XA (forward) or s*G (backward), [M,R] bf16
  o = align256(o + rows * L.R * 2);
  L.off_g = o;  // G [M,R] bf16 (backward)
  o = align256(o + rows * L.R * 2);
  L.total = o;
  return L;
}

// ---------------------------------------------------------------------------
// Argument checks
// ---------------------------------------------------------------------------
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

qlora_status check_w(const qlora_w4* w) {
  if (!w || !w->idx || !w->absmax || !w->codebook) return QLORA_ERR_INVALID_ARG;
  if (w->N < 0 || w->K < 0 || w->block != 64) return QLORA_ERR_INVALID_ARG;
  if (w->K % 64 != 0) return QLORA_ERR_UNSUPPORTED;
  if (!al16(w->idx) || !al16(w->absmax) || !al16(w->codebook)) return QLORA_ERR_ALIGNMENT;
  return QLORA_OK;
}

struct Segs {
  int32_t n;
  int32_t start[kMaxSeg + 1];
};

qlora_status check_layer(int64_t M, const qlora_w4* W, int32_t r, int32_t n_seg, const int64_t* seg_n, Segs* sg) {
  qlora_status st = check_w(W);
  if (st != QLORA_OK) return st;
  if (M < 0) return QLORA_ERR_INVALID_ARG;
  if (W->N < 8 || W->K < 64) return QLORA_ERR_INVALID_ARG;
  if (W->N % 8 != 0) return QLORA_ERR_UNSUPPORTED;
  if (W->N > (int64_t(1) << 30) || W->K > (int64_t(1) << 30) || M > (int64_t(1) << 30))
    return QLORA_ERR_UNSUPPORTED;
  if (r < 8 || r > 128 || r % 8 != 0) return QLORA_ERR_INVALID_ARG;
  if (n_seg < 1 || n_seg > kMaxSeg) return QLORA_ERR_INVALID_ARG;
  if (int64_t(n_seg) * r > 256) return QLORA_ERR_UNSUPPORTED;
  if (n_seg > 1 && !seg_n) return QLORA_ERR_INVALID_ARG;
  sg->n = n_seg;
  int64_t off = 0;
  sg->start[0] = 0;
  for (int j = 0; j < n_seg; ++j) {
    const int64_t w = (n_seg == 1 && !seg_n) ? W->N : seg_n[j];
    if (w <= 0) return QLORA_ERR_INVALID_ARG;
    if (j < n_seg - 1 && w % 128 != 0) return QLORA_ERR_UNSUPPORTED;
    off += w;
    sg->start[j + 1] = static_cast<int32_t>(off);
  }
  if (off != W->N) return QLORA_ERR_INVALID_ARG;
  return QLORA_OK;
}

qlora_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA; }

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------
// L2 policy bits for the large GEMMs (GemmArgs::l2_hints); QLORA_L2_HINTS
// overrides the default.
int l2_hints() {
  static const int v = [] {
    const char* e = std::getenv("QLORA_L2_HINTS");
    return e ? std::atoi(e) : 7;
  }();
  return v;
}

// Band of the pair GEMM's tile order (GemmArgs::group_m).  Both operands
// have 256 rows per tile, so a tile of either is 256*K*2 bytes.  A band holds
// as many tiles of one operand as fit in `budget` bytes of L2 (at least 8);
// the other operand is then read once per band.  Modelled DRAM reads, in tiles:
//   row bands:    ceil(m_tiles/g)*n_tiles + m_tiles
//   column bands: ceil(n_tiles/g)*m_tiles + n_tiles
// and the smaller wins.  QLORA_GROUP_M forces a band (signed as group_m),
// QLORA_BAND_MB sets the budget.
int pair_group(int64_t m_tiles, int64_t n_tiles, int64_t K) {
  static const int forced = [] {
    const char* e = std::getenv("QLORA_GROUP_M");
    return e ? std::atoi(e) : 0;
  }();
  static const int64_t budget = [] {
    const char* e = std::getenv("QLORA_BAND_MB");
    const int64_t mb = e ? std::atoll(e) : 32;
    return (mb > 0 ? mb : 32) << 20;
  }();
  if (forced != 0) return forced;
  const int64_t tile_bytes = 256 * K * 2;
  // At least 8 tiles per band: with 7.3 MB tiles (K = 14336) a wave's operands
  // exceed L2 anyway, and bands of 8 measured best there (+0.6% on the MLP
  // step against bands of 4; bands of 6 and row bands of 6 or 8 in between).
  const int64_t g = std::max<int64_t>(8, budget / std::max<int64_t>(tile_bytes, 1));
  const int64_t rows = cdiv(m_tiles, g) * n_tiles + m_tiles;
  const int64_t cols = cdiv(n_tiles, g) * m_tiles + n_tiles;
  const int64_t gi = std::min<int64_t>(g, 1 << 20);
  return rows <= cols ? static_cast<int>(gi) : -static_cast<int>(gi);
}

constexpr int kSmemLimit = 232448;

// Launches may overlap the tail of their predecessor in the stream
// (programmatic dependent launch; each kernel waits with griddepcontrol.wait
// before it touches global memory, so the overlap covers only its prologue:
// barrier set-up, tensor-memory allocation, descriptor prefetch).  On by
// default; QLORA_PDL=0 turns it off.
bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("QLORA_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct TileCfg {
  int bn, stages;
  uint32_t stage_bytes;
  size_t smem;
};

// Split-sum buffer inside the idle ring when each cluster has one tile
// (QLORA_RED_IN_RING=0 turns it off).
bool red_in_ring_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("QLORA_RED_IN_RING");
    return !(e && e[0] == '0');
  }();
  return on;
}

// Ring depth cap of the rank-r GEMMs (QLORA_RED_STAGES overrides; 2..10).
int red_stage_cap() {
  static const int v = [] {
    const char* e = std::getenv("QLORA_RED_STAGES");
    const int n = e ? std::atoi(e) : kMaxStages;
    return std::max(2, std::min(kMaxStages, n));
  }();
  return v;
}

// Ring geometry of gemm_tc_kernel; `red` reserves the split-sum buffer after
// the ring, `in_ring` puts it inside the ring instead (one tile per cluster).
TileCfg tile_cfg(int bn, bool red = false, bool in_ring = false) {
  TileCfg c;
  c.bn = bn;
  c.stage_bytes = static_cast<uint32_t>(rup(kATileBytes + int64_t(bn) * 128, 1024));
  const int64_t extra = (red && !in_ring) ? kRedBytes : 0;
  const int64_t ring = red ? int64_t(kSmemLimit) - extra - 1024 - 256 : 200 * 1024;
  c.stages = std::min<int>(red ? red_stage_cap() : 8, static_cast<int>(ring / c.stage_bytes));
  if (in_ring && int64_t(c.stages) * c.stage_bytes < int64_t(kRedBytes)) c.stages = 0;  // caller falls back
  c.smem = size_t(c.stages) * c.stage_bytes + extra + 1024 + 256;
  return c;
}

template <bool A_MN, bool B_MN, int EPI>
qlora_status launch_gemm(const char* name, dim3 grid, const TileCfg& tc, const CUtensorMap& a, const CUtensorMap& b,
                         const CUtensorMap& a2, const CUtensorMap& b2, GemmArgs args, cudaStream_t st) {
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(attr_once[dev & 63], [] {
    cudaFuncSetAttribute(gemm_tc_kernel<A_MN, B_MN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  });
  args.bn = tc.bn;
  args.stages = tc.stages;
  args.stage_bytes = tc.stage_bytes;
  args.timeout_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  args.debug_stall = take_stall(name) ? 1 : 0;
  args.l2_hints = (EPI == EPI_BF16) ? (l2_hints() & 1) : 0;
  // `grid` is the tile grid; the kernel is persistent with one CTA per SM.
  args.m_tiles = static_cast<int32_t>(grid.x);
  args.n_tiles = static_cast<int32_t>(grid.y);
  args.z_tiles = static_cast<int32_t>(grid.z);
  const int64_t tiles = int64_t(grid.x) * grid.y * grid.z;
  const unsigned ctas = static_cast<unsigned>(std::min<int64_t>(tiles, sm_count(dev)));
  cudaError_t e;
  {
    LaunchScope ls(name, st);
    GemmArgs none;
    std::memset(&none, 0, sizeof(none));
    e = launch_k(gemm_tc_kernel<A_MN, B_MN, EPI>, dim3(ctas), dim3(192), tc.smem, st, a, b, a2, b2, args, none);
  }
  return cuda_status(e);
}

// Clusters of `splits` CTAs of gemm_tc_kernel<.., EPI_RED> that fit on the
// device at once (cached per instance, device and cluster size).
template <bool A_MN, bool B_MN>
int max_red_clusters(int splits, size_t smem) {
  static std::mutex mu;
  static int cache[64][kMaxSplits + 1] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  int& c = cache[dev & 63][splits];
  if (c == 0) {
    auto kern = gemm_tc_kernel<A_MN, B_MN, EPI_RED>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(splits) * 64u);
    cfg.blockDim = dim3(kRedThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = sm_count(dev) / splits;
    }
    c = std::max(1, n);
  }
  return c;
}

// Splits (cluster size) for an EPI_RED GEMM with `tiles` output tiles of
// `nkb` 64-wide reduction blocks: the most splits, up to 8, for which all
// clusters of one wave fit on the device at once.
template <bool A_MN, bool B_MN>
int red_splits(int64_t tiles, int64_t nkb, size_t smem) {
  static const int64_t most = [] {  // QLORA_RED_MAX_SPLITS caps the cluster size (1..8)
    const char* e = std::getenv("QLORA_RED_MAX_SPLITS");
    const int64_t n = e ? std::atoll(e) : kMaxSplits;
    return std::max<int64_t>(1, std::min<int64_t>(kMaxSplits, n));
  }();
  const int64_t cap = std::min<int64_t>({most, std::max<int64_t>(1, nkb),
                                         std::max<int64_t>(1, int64_t(sm_count(cur_dev())) / std::max<int64_t>(tiles, 1))});
  for (int64_t sp = cap; sp > 1; --sp)
    if (max_red_clusters<A_MN, B_MN>(static_cast<int>(sp), smem) >= tiles) return static_cast<int>(sp);
  return 1;
}

// One problem of a gemm_tc_kernel<.., EPI_RED> launch: tiles m_tiles x
// n_tiles x zseg (zseg adapter segments for GM_G, else 1) of g.tile_m rows.
struct RedProb {
  GemmArgs g;
  CUtensorMap a, b;
  int64_t m_tiles, n_tiles, zseg;
  int bn;
};

// Row-tile height of a rank-r GEMM with a K-major A operand (XA, G) and
// `splits` CTAs per tile: 128 rows, or -- when 128-row tiles leave clusters
// of the wave unused -- the smallest multiple of 8 (at least 64) whose tiles
// still fit in one wave, so that more SMs stream the operand.  Every row's
// sum is over the same reduction chunks in the same order either way.
// QLORA_RED_TILE_M=0 keeps 128 (read on every call).
template <bool B_MN>
int red_tile_m(int64_t M, int64_t zseg, int splits, size_t smem) {
  const char* e = std::getenv("QLORA_RED_TILE_M");
  if (e && e[0] == '0') return 128;
  const int64_t per_seg = max_red_clusters<false, B_MN>(splits, smem) / std::max<int64_t>(zseg, 1);
  if (per_seg <= cdiv(M, 128)) return 128;
  const int64_t tm = std::max<int64_t>(64, rup(cdiv(M, per_seg), 8));
  return (tm < 128 && cdiv(M, tm) > cdiv(M, 128)) ? static_cast<int>(tm) : 128;
}

// gemm_tc_kernel<.., EPI_RED>: `splits` CTAs per tile in one cluster; an
// optional second problem shares the launch (its tiles follow the first's).
template <bool A_MN, bool B_MN>
qlora_status launch_gemm_red(const char* name, int splits, const TileCfg& tc_in, RedProb p1, const RedProb* p2,
                             cudaStream_t st) {
  auto kern = gemm_tc_kernel<A_MN, B_MN, EPI_RED>;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(attr_once[dev & 63], [kern] {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  });
  const int64_t tiles = p1.m_tiles * p1.n_tiles * p1.zseg + (p2 ? p2->m_tiles * p2->n_tiles * p2->zseg : 0);
  const int64_t clusters = std::min<int64_t>(tiles, max_red_clusters<A_MN, B_MN>(splits, tc_in.smem));
  // One tile per cluster: the split-sum buffer can share the ring, which then
  // gets the 34 KB the buffer would occupy (QLORA_RED_IN_RING=0 keeps them apart).
  const TileCfg ring_tc = tile_cfg(tc_in.bn, true, true);
  const bool in_ring = tiles <= clusters && ring_tc.stages > tc_in.stages && red_in_ring_enabled();
  const TileCfg& tc = in_ring ? ring_tc : tc_in;
  auto fill = [&](RedProb& pr) {
    GemmArgs& a = pr.g;
    a.bn = pr.bn;
    a.stages = tc.stages;
    a.stage_bytes = tc.stage_bytes;
    a.timeout_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    a.l2_hints = 0;
    a.splits = splits;
    a.red_in_ring = in_ring ? 1 : 0;
    a.m_tiles = static_cast<int32_t>(pr.m_tiles);
    a.n_tiles = static_cast<int32_t>(pr.n_tiles);
    a.z_tiles = static_cast<int32_t>(pr.zseg * splits);
  };
  fill(p1);
  p1.g.debug_stall = take_stall(name) ? 1 : 0;
  RedProb q2;
  if (p2) {
    q2 = *p2;
    fill(q2);
  } else {
    std::memset(&q2.g, 0, sizeof(q2.g));
    q2.a = p1.a;
    q2.b = p1.b;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * splits));
  cfg.blockDim = dim3(kRedThreads);
  cfg.dynamicSmemBytes = tc.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e;
  {
    LaunchScope ls(name, st);
    e = cudaLaunchKernelEx(&cfg, kern, p1.a, p1.b, q2.a, q2.b, p1.g, q2.g);
  }
  return cuda_status(e);
}

// Splits of XA = X.A: shared by the forward and the static-scratch entry
// point so both sum the same reduction chunks in the same order.
int xa_splits(int64_t M, int64_t K, int64_t R) {
  const TileCfg tc = tile_cfg(static_cast<int>(rup(R, 64)), true);
  return red_splits<false, true>(cdiv(M, 128), K / 64, tc.smem);
}

// CTA-pair kernel for the two large GEMMs (256 x 256 tiles, K-major operands).
constexpr int kPairStages = 6;

bool pair_enabled() {
  const char* e = std::getenv("QLORA_DISABLE_PAIR");
  return !(e && e[0] == '1');
}

// In-kernel dequantisation in the pair GEMM (the 4-bit weight expanded into
// the B tiles, no dequantised copy in the workspace).  QLORA_FUSED_DQ=1 turns
// it on, =0 off.
// Read on every call (not cached), so one process can run both paths.
bool fused_dq_enabled() {
  const char* e = std::getenv("QLORA_FUSED_DQ");
  return e && e[0] == '1';
}

// The row-major Wd written by the rank-r GEMM launch that precedes its use
// (XA in the forward, G in the backward) instead of a dequantiser launch of
// its own.  Measured on GB300 (whole step, interleaved): faster at M = 8192
// tokens (Llama-3-8B MLP +2.3%, the two-adapter gate/up call +1.6%, fused QKV
// +1.1%), slower at M = 4096 (q_proj -2.1%) and M = 256 (-6.8%), where the
// separate dequantiser's small CTAs overlap the neighbouring launches better
// than one launch of full-SM CTAs.  So: from 8192 tokens on.
// QLORA_DQ_IN_RANKR=0 / =1 forces either way (read on every call).
constexpr int64_t kDqInRankrMinM = 8192;
bool dq_in_rankr_enabled(int64_t M) {
  const char* e = std::getenv("QLORA_DQ_IN_RANKR");
  if (e && e[0] == '0') return false;
  if (e && e[0] == '1') return true;
  return M >= kDqInRankrMinM;
}

// Attach the dequantisation of W into the row-major Wd to a rank-r launch.
void attach_dequant(GemmArgs& g, const qlora_w4* W, void* Wd) {
  g.codebook = W->codebook;
  g.dq_idx = static_cast<const uint8_t*>(W->idx);
  g.dq_absmax = W->absmax;
  g.dq_out = static_cast<__nv_bfloat16*>(Wd);
  g.dq_words = W->N * W->K / 8;
}

template <bool B_MN, bool FUSED>
qlora_status launch_gemm_pair(const char* name, int64_t m_tiles, int64_t n_tiles, const CUtensorMap& a,
                              const CUtensorMap& b, const CUtensorMap& a2, const CUtensorMap& b2, GemmArgs args,
                              cudaStream_t st) {
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  const int stages = kPairStages;
  const size_t smem = size_t(stages) * kPairStageBytes + (FUSED ? kDqSlots * kDqSlotBytes : 0) + 1024 + 512;
  std::call_once(attr_once[dev & 63], [smem] {
    cudaFuncSetAttribute(gemm_pair_kernel<B_MN, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
  });
  args.bn = 256;
  args.stages = stages;
  args.stage_bytes = kPairStageBytes;
  args.timeout_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  args.debug_stall = take_stall(name) ? 1 : 0;
  args.l2_hints = l2_hints();
  args.group_m = pair_group(m_tiles, n_tiles, args.red_len);
  args.m_tiles = static_cast<int32_t>(m_tiles);
  args.n_tiles = static_cast<int32_t>(n_tiles);
  args.z_tiles = 1;
  const int64_t pairs = std::min<int64_t>(m_tiles * n_tiles, sm_count(dev) / 2);
  cudaError_t e;
  {
    LaunchScope ls(name, st);
    e = launch_k(gemm_pair_kernel<B_MN, FUSED>, dim3(static_cast<unsigned>(2 * pairs)),
                 dim3(FUSED ? 192 + 32 * kDqWarps : 192), smem, st, a, b, a2, b2, args);
  }
  return cuda_status(e);
}

GemmArgs base_args(uint32_t* err) {
  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  g.splits = 1;
  g.nseg = 1;
  g.tile_m = 128;
  g.err = err;
  return g;
}

qlora_status launch_dequant(const qlora_w4* w, void* out_bf16, float* out_f32, cudaStream_t st) {
  const int64_t groups = w->N * w->K / 8;
  if (groups == 0) return QLORA_OK;
  const int64_t blocks = std::min<int64_t>(cdiv(groups, 1024), int64_t(kSMs) * 8);  // 8 warps x 128 groups
  LaunchScope ls("dequant4", st);
  return cuda_status(launch_k(dequant4_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                              reinterpret_cast<const uint32_t*>(w->idx), w->absmax, w->codebook, groups,
                              reinterpret_cast<uint4*>(out_bf16), reinterpret_cast<float4*>(out_f32)));
}

TransposeJob tjob(const void* src, int64_t rows, int64_t cols, int64_t lds, void* dst, int64_t drows, int64_t dcols,
                  int64_t ldd) {
  TransposeJob j;
  j.src = reinterpret_cast<const __nv_bfloat16*>(src);
  j.dst = reinterpret_cast<__nv_bfloat16*>(dst);
  j.rows = static_cast<int32_t>(rows);
  j.cols = static_cast<int32_t>(cols);
  j.dst_rows = static_cast<int32_t>(drows);
  j.dst_cols = static_cast<int32_t>(dcols);
  j.lds = lds;
  j.ldd = ldd;
  return j;
}

// One launch for up to three transposes (tiles of all jobs in one flat grid).
qlora_status launch_transposes(const char* name, const TransposeJob* jobs, int n, cudaStream_t st) {
  TransposeJobs tj;
  std::memset(&tj, 0, sizeof(tj));
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {
    tj.job[i] = jobs[i];
    tj.job[i].tiles_x = static_cast<int32_t>(cdiv(jobs[i].dst_cols, 32));
    tj.job[i].tile_begin = static_cast<int32_t>(total);
    total += cdiv(jobs[i].dst_cols, 32) * cdiv(jobs[i].dst_rows, 32);
  }
  tj.njobs = n;
  if (total == 0) return QLORA_OK;
  LaunchScope ls(name, st);
  return cuda_status(launch_k(transpose_jobs_kernel, dim3(static_cast<unsigned>(total)), dim3(256), 0, st, tj));
}

qlora_status launch_reduce(const char* name, const ReduceArgs& ra, cudaStream_t st) {
  if (int64_t(ra.rows) * ra.cols == 0) return QLORA_OK;
  dim3 grid(static_cast<unsigned>(cdiv(ra.rows, 32)), static_cast<unsigned>(cdiv(ra.cols, 32)));
  LaunchScope ls(name, st);
  return cuda_status(launch_k(reduce_tile_kernel, grid, dim3(256), 0, st, ra));
}

ReduceArgs reduce_args(const float* part, int splits, int64_t rows, int64_t cols, int64_t ld, int64_t sstride,
                       float scale) {
  ReduceArgs ra;
  std::memset(&ra, 0, sizeof(ra));
  ra.part = part;
  ra.splits = splits;
  ra.rows = static_cast<int32_t>(rows);
  ra.cols = static_cast<int32_t>(cols);
  ra.ld = ld;
  ra.sstride = sstride;
  ra.scale = scale;
  return ra;
}

#define QL_TRY(expr)                  \
  do {                                \
    qlora_status _s = (expr);         \
    if (_s != QLORA_OK) return _s;    \
  } while (0)

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

const char* qlora_status_str(qlora_status s) {
  switch (s) {
    case QLORA_OK: return "ok";
    case QLORA_ERR_INVALID_ARG: return "invalid argument";
    case QLORA_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case QLORA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case QLORA_ERR_WORKSPACE: return "workspace missing or too small";
    case QLORA_ERR_CUDA: return "CUDA error";
    case QLORA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

void qlora_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(std::max<uint64_t>(ns, 1000000ull)); }

void qlora_debug_stall_next_launch(const char* label) {
  std::lock_guard<std::mutex> lk(g_stall_mu);
  g_stall_label[0] = 0;
  if (label) {
    std::strncpy(g_stall_label, label, sizeof(g_stall_label) - 1);
    g_stall_label[sizeof(g_stall_label) - 1] = 0;
  }
}

void qlora_profiler_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
}

uint64_t qlora_launch_counter(void) { return g_launches.load(); }

int qlora_profiler_collect(qlora_kernel_stat* out, int max_entries) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_prof_recs);
  }
  std::vector<qlora_kernel_stat> stats;
  for (const ProfRec& pr : recs) {
    cudaEventSynchronize(pr.b);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, pr.a, pr.b);
    auto itr = std::find_if(stats.begin(), stats.end(),
                            [&](const qlora_kernel_stat& k) { return std::strcmp(k.name, pr.name) == 0; });
    if (itr == stats.end()) {
      stats.push_back({pr.name, 1, static_cast<double>(ms)});
    } else {
      itr->launches += 1;
      itr->total_ms += ms;
    }
  }
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (const ProfRec& pr : recs) {
      g_event_pool.push_back(pr.a);
      g_event_pool.push_back(pr.b);
    }
  }
  for (int i = 0; i < static_cast<int>(stats.size()) && i < max_entries && out; ++i) out[i] = stats[i];
  return static_cast<int>(stats.size());
}

size_t qlora_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r, int32_t n_seg) {
  if (M < 0 || N <= 0 || K <= 0 || r <= 0 || n_seg <= 0) return 0;
  return layout(M, N, K, r, n_seg).total;
}

qlora_status qlora_check_device_error(void* ws, cudaStream_t st) {
  if (!ws) return QLORA_ERR_WORKSPACE;
  if (cudaStreamSynchronize(st) != cudaSuccess) return QLORA_ERR_CUDA;
  uint32_t flag = 0;
  if (cudaMemcpy(&flag, ws, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return QLORA_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return QLORA_ERR_CUDA;
  if (flag != 0) {
    if (cudaMemset(ws, 0, 4) != cudaSuccess) return QLORA_ERR_CUDA;
    return QLORA_ERR_TIMEOUT;
  }
  return QLORA_OK;
}

qlora_status dequant_4bit(const qlora_w4* w, void* out_bf16, float* out_f32, cudaStream_t st) {
  QL_TRY(check_w(w));
  if (!out_bf16 && !out_f32) return QLORA_ERR_INVALID_ARG;
  if ((out_bf16 && !al16(out_bf16)) || (out_f32 && !al16(out_f32))) return QLORA_ERR_ALIGNMENT;
  return launch_dequant(w, out_bf16, out_f32, st);
}

qlora_status quantize_4bit(const void* W, int32_t w_is_bf16, int64_t N, int64_t K, const float* codebook,
                           uint8_t* idx, float* absmax, cudaStream_t st) {
  if (N < 0 || K <= 0) return QLORA_ERR_INVALID_ARG;
  if (K % 64 != 0) return QLORA_ERR_UNSUPPORTED;
  if (N == 0) return QLORA_OK;
  if (!W || !codebook || !idx || !absmax) return QLORA_ERR_INVALID_ARG;
  if (!al16(W) || !al16(idx) || !al16(absmax)) return QLORA_ERR_ALIGNMENT;
  const int64_t groups = N * K / 8;
  // one wave of one 1024-thread CTA per SM: each SM builds its table once
  const int64_t blocks = std::min<int64_t>(cdiv(groups, 1024), int64_t(sm_count(cur_dev())));
  LaunchScope ls("quantize4", st);
  cudaError_t e;
  if (w_is_bf16)
    e = launch_k(quantize4_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(1024), 0, st, W, codebook, groups,
                 reinterpret_cast<uint32_t*>(idx), absmax);
  else
    e = launch_k(quantize4_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(1024), 0, st, W, codebook, groups,
                 reinterpret_cast<uint32_t*>(idx), absmax);
  return cuda_status(e);
}

qlora_status qlora_linear_fwd(const void* X, int64_t M, const qlora_w4* W, const void* A, const void* B, int32_t r,
                              int32_t n_seg, const int64_t* seg_n, float s, void* Y, void* XA_save, void* ws,
                              size_t ws_bytes, cudaStream_t st) {
  Segs sg;
  QL_TRY(check_layer(M, W, r, n_seg, seg_n, &sg));
  if (!X || !A || !B || !Y || !XA_save) return QLORA_ERR_INVALID_ARG;
  if (!al16(X) || !al16(A) || !al16(B) || !al16(Y) || !al16(XA_save)) return QLORA_ERR_ALIGNMENT;
  const int64_t N = W->N, K = W->K;
  const Layout L = layout(M, N, K, r, n_seg);
  if (!ws) return QLORA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return QLORA_ERR_ALIGNMENT;
  if (ws_bytes < L.total) return QLORA_ERR_WORKSPACE;
  if (M == 0) return QLORA_OK;
  if (!encode_fn()) return QLORA_ERR_CUDA;

  uint8_t* w8 = static_cast<uint8_t*>(ws);
  uint32_t* err = reinterpret_cast<uint32_t*>(w8 + L.off_err);
  void* Wd = w8 + L.off_wd;
  void* Bt = w8 + L.off_bt;
  void* XAs = w8 + L.off_xas;
  const int64_t R = L.R;

  // 1. B^T [N,Rp] (zero columns r..Rp-1): the rank-r B-operand of the
  //    single-CTA Y GEMM (the CTA-pair kernel reads B [r,N] MN-major)
  bool b256 = true;
  for (int j = 1; j < n_seg; ++j)
    if (sg.start[j] % 256 != 0) b256 = false;
  const bool pair_fwd = b256 && pair_enabled();
  if (!pair_fwd) {
    const TransposeJob jobs[1] = {tjob(B, r, N, N, Bt, N, L.Rp, L.Rp)};
    QL_TRY(launch_transposes("transpose_B", jobs, 1, st));
  }

  // 2. Wd = deq(W), unless the pair GEMM dequantises in shared memory
  const bool fused_fwd = pair_fwd && fused_dq_enabled();
  const bool dq_in_xa = !fused_fwd && dq_in_rankr_enabled(M);
  if (!fused_fwd && !dq_in_xa) QL_TRY(launch_dequant(W, Wd, nullptr, st));

  // 3. XA = X . A (A read MN-major; splits of K summed in the kernel);
  //    writes XA_save = bf16(XA) and s*XA
  CUtensorMap mX, mWd, mXAs, mBt;
  if (!make_map(&mX, X, K, M, K, 128)) return QLORA_ERR_CUDA;  // 128-row boxes of the base GEMM
  {
    CUtensorMap mA, mXr;
    const TileCfg tc = tile_cfg(static_cast<int>(rup(R, 64)), true);
    const int splits = xa_splits(M, K, R);
    const int tm = red_tile_m<true>(M, 1, splits, tc.smem);
    if (!make_map(&mXr, X, K, M, K, static_cast<uint32_t>(tm)) || !make_map(&mA, A, R, K, R, 64))
      return QLORA_ERR_CUDA;
    GemmArgs g = base_args(err);
    g.tile_m = tm;
    g.M = static_cast<int32_t>(M);
    g.N = static_cast<int32_t>(R);
    g.mode = GM_PLAIN;
    g.red_len = static_cast<int32_t>(K);
    g.out_valid = static_cast<int32_t>(R);
    g.red_scale = s;
    g.red_bf16 = reinterpret_cast<__nv_bfloat16*>(XA_save);
    g.red_bf16_s = reinterpret_cast<__nv_bfloat16*>(XAs);
    g.red_ld = R;
    if (dq_in_xa) attach_dequant(g, W, Wd);  // the Wd of step 4
    QL_TRY((launch_gemm_red<false, true>("gemm_xa", splits, tc, RedProb{g, mXr, mA, cdiv(M, tm), 1, 1, tc.bn},
                                         nullptr, st)));
  }

  // 4. Y = X . Wd^T + (s XA) . B
  {
    const bool pair = pair_fwd;
    const int bn = b256 ? 256 : 128;
    const TileCfg tc = tile_cfg(bn);
    const uint32_t brows = pair ? 128u : static_cast<uint32_t>(bn);  // rows of B staged per CTA
    if (fused_fwd) {
      mWd = mX;  // unused: the kernel reads the 4-bit weight itself
    } else {
      if (!make_map(&mWd, Wd, K, N, K, brows)) return QLORA_ERR_CUDA;
    }
    if (!make_map(&mXAs, XAs, R, M, R, 128)) return QLORA_ERR_CUDA;
    if (pair ? !make_map(&mBt, B, N, r, N, 64) : !make_map(&mBt, Bt, L.Rp, N, L.Rp, brows)) return QLORA_ERR_CUDA;
    GemmArgs g = base_args(err);
    g.M = static_cast<int32_t>(M);
    g.N = static_cast<int32_t>(N);
    g.mode = GM_FWD;
    g.red_len = static_cast<int32_t>(K);
    g.r = r;
    g.nseg = n_seg;
    for (int j = 0; j <= n_seg; ++j) g.seg_start[j] = sg.start[j];
    g.lora_ksteps = static_cast<int32_t>(L.Rp / 16);
    g.lora_atoms = static_cast<int32_t>(cdiv(L.Rp, 64));
    g.out_ld = static_cast<int32_t>(N);
    g.out_valid = static_cast<int32_t>(N);
    g.out = Y;
    g.codebook = W->codebook;
    g.dq_idx = W->idx;
    g.dq_absmax = W->absmax;
    g.dq_k = static_cast<int32_t>(K);
    if (fused_fwd) {
      QL_TRY((launch_gemm_pair<false, true>("gemm_fwd", cdiv(M, 256), cdiv(N, 256), mX, mWd, mXAs, mBt, g, st)));
    } else if (pair) {
      QL_TRY((launch_gemm_pair<false, false>("gemm_fwd", cdiv(M, 256), cdiv(N, 256), mX, mWd, mXAs, mBt, g, st)));
    } else {
      dim3 grid(static_cast<unsigned>(cdiv(M, 128)), static_cast<unsigned>(cdiv(N, bn)), 1);
      QL_TRY((launch_gemm<false, false, EPI_BF16>("gemm_fwd", grid, tc, mX, mWd, mXAs, mBt, g, st)));
    }
  }
  return QLORA_OK;
}

}  // extern "C"

namespace {
// Backward; `accumulate` adds the adapter gradients into dA and dB.
qlora_status linear_bwd(const void* dY, const void* X, const void* XA_saved, int64_t M, const qlora_w4* W,
                        const void* A, const void* B, int32_t r, int32_t n_seg, const int64_t* seg_n, float s,
                        void* dX, float* dA, float* dB, void* ws, size_t ws_bytes, cudaStream_t st, bool accumulate) {
  Segs sg;
  QL_TRY(check_layer(M, W, r, n_seg, seg_n, &sg));
  if (!dY || !X || !XA_saved || !A || !B || !dA || !dB) return QLORA_ERR_INVALID_ARG;
  if (!al16(dY) || !al16(X) || !al16(XA_saved) || !al16(A) || !al16(B) || !al16(dA) || !al16(dB) ||
      (dX && !al16(dX)))
    return QLORA_ERR_ALIGNMENT;
  const int64_t N = W->N, K = W->K;
  const Layout L = layout(M, N, K, r, n_seg);
  if (!ws) return QLORA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return QLORA_ERR_ALIGNMENT;
  if (ws_bytes < L.total) return QLORA_ERR_WORKSPACE;
  const int64_t R = L.R;
  if (M == 0) {
    if (accumulate) return QLORA_OK;  // nothing to add
    QL_TRY(cuda_status(cudaMemsetAsync(dA, 0, size_t(K) * R * 4, st)));
    QL_TRY(cuda_status(cudaMemsetAsync(dB, 0, size_t(r) * N * 4, st)));
    return QLORA_OK;
  }
  if (!encode_fn()) return QLORA_ERR_CUDA;

  uint8_t* w8 = static_cast<uint8_t*>(ws);
  uint32_t* err = reinterpret_cast<uint32_t*>(w8 + L.off_err);
  void* WdT = w8 + L.off_wd;
  void* Gs = w8 + L.off_xas;
  void* G = w8 + L.off_g;

  CUtensorMap mdY, mB, mWdT, mGs, mA, mXmn, mGmn, mdYmn, mXAmn;
  if (!make_map(&mdY, dY, N, M, N, 128)) return QLORA_ERR_CUDA;  // 128-row boxes of the base GEMM
  // the pair dX reads the row-major Wd; the G launch writes it when enabled
  const bool dx_pair = dX && pair_enabled();
  const bool dx_fused = dx_pair && fused_dq_enabled();
  const bool dq_in_g = dx_pair && !dx_fused && dq_in_rankr_enabled(M);

  // 1. G = dY . B^T per segment (splits of the segment's columns summed in
  //    the kernel); writes s*G and G
  {
    const int bn = static_cast<int>(rup(r, 16));
    const TileCfg tc = tile_cfg(bn, true);
    const int64_t mt = cdiv(M, 128);
    int64_t min_nkb = INT64_MAX;
    for (int j = 0; j < n_seg; ++j) min_nkb = std::min<int64_t>(min_nkb, cdiv(sg.start[j + 1] - sg.start[j], 64));
    const int splits = red_splits<false, false>(mt * n_seg, min_nkb, tc.smem);
    const int tm = red_tile_m<false>(M, n_seg, splits, tc.smem);
    CUtensorMap mdYr;
    if (!make_map(&mdYr, dY, N, M, N, static_cast<uint32_t>(tm)) || !make_map(&mB, B, N, r, N, static_cast<uint32_t>(bn)))
      return QLORA_ERR_CUDA;
    GemmArgs g = base_args(err);
    g.tile_m = tm;
    g.M = static_cast<int32_t>(M);
    g.N = r;
    g.mode = GM_G;
    g.r = r;
    g.nseg = n_seg;
    for (int j = 0; j <= n_seg; ++j) g.seg_start[j] = sg.start[j];
    g.out_valid = r;
    g.red_scale = s;
    g.red_bf16 = reinterpret_cast<__nv_bfloat16*>(G);
    g.red_bf16_s = reinterpret_cast<__nv_bfloat16*>(Gs);
    g.red_ld = R;
    if (dq_in_g) attach_dequant(g, W, WdT);  // the row-major Wd of step 2
    QL_TRY((launch_gemm_red<false, false>("gemm_g", splits, tc, RedProb{g, mdYr, mB, cdiv(M, tm), 1, n_seg, bn},
                                          nullptr, st)));
  }

  // 2. dX = dY . Wd + (s G) . A^T
  if (dX) {
    const bool pair = dx_pair;
    const bool fused = dx_fused;
    const int bn = 256;
    const TileCfg tc = tile_cfg(bn);
    if (fused) {
      // the pair kernel expands the 4-bit codes into its MN-major B tiles
      mWdT = mdY;  // unused
    } else if (pair) {
      // row-major Wd [N,K], read MN-major by the pair kernel
      if (!dq_in_g) QL_TRY(launch_dequant(W, WdT, nullptr, st));
      if (!make_map(&mWdT, WdT, K, N, K, 64)) return QLORA_ERR_CUDA;
    } else {
      dim3 grid(static_cast<unsigned>(K / 64), static_cast<unsigned>(cdiv(N, 64)));
      {
        LaunchScope ls("dequant4_t", st);
        QL_TRY(cuda_status(launch_k(dequant4_t_kernel, grid, dim3(256), 0, st, W->idx, W->absmax, W->codebook,
                                    static_cast<int32_t>(N), static_cast<int32_t>(K),
                                    reinterpret_cast<__nv_bfloat16*>(WdT), N)));
      }
      if (!make_map(&mWdT, WdT, N, K, N, static_cast<uint32_t>(bn))) return QLORA_ERR_CUDA;
    }
    const uint32_t brows = pair ? 128u : static_cast<uint32_t>(bn);
    if (!make_map(&mGs, Gs, R, M, R, 128) || !make_map(&mA, A, R, K, R, brows)) return QLORA_ERR_CUDA;
    GemmArgs g = base_args(err);
    g.M = static_cast<int32_t>(M);
    g.N = static_cast<int32_t>(K);
    g.mode = GM_DX;
    g.red_len = static_cast<int32_t>(N);
    g.r = r;
    g.nseg = n_seg;
    g.lora_ksteps = static_cast<int32_t>(cdiv(R, 16));
    g.lora_atoms = static_cast<int32_t>(cdiv(R, 64));
    g.out_ld = static_cast<int32_t>(K);
    g.out_valid = static_cast<int32_t>(K);
    g.out = dX;
    g.codebook = W->codebook;
    g.dq_idx = W->idx;
    g.dq_absmax = W->absmax;
    g.dq_k = static_cast<int32_t>(K);
    if (fused) {
      QL_TRY((launch_gemm_pair<true, true>("gemm_dx", cdiv(M, 256), cdiv(K, 256), mdY, mWdT, mGs, mA, g, st)));
    } else if (pair) {
      QL_TRY((launch_gemm_pair<true, false>("gemm_dx", cdiv(M, 256), cdiv(K, 256), mdY, mWdT, mGs, mA, g, st)));
    } else {
      dim3 grid(static_cast<unsigned>(cdiv(M, 128)), static_cast<unsigned>(cdiv(K, bn)), 1);
      QL_TRY((launch_gemm<false, false, EPI_BF16>("gemm_dx", grid, tc, mdY, mWdT, mGs, mA, g, st)));
    }
  }

  // 3+4. dA = s X^T G and dB = s XA^T dY in one launch (both reduce over the
  //    M tokens and read every operand MN-major; splits of M summed in the
  //    kernel).  dB is computed as dB^T = dY^T . XA and stored transposed.
  //    A dA tile streams 128 columns of X, a dB tile 128 columns of dY: the
  //    tiles of the two problems are the same amount of work.
  {
    const int bn_a = static_cast<int>(rup(R, 64)), bn_b = static_cast<int>(rup(r, 64));
    const TileCfg tc = tile_cfg(std::max(bn_a, bn_b), true);
    const int64_t kt = cdiv(K, 128), nt = cdiv(N, 128);
    const int splits = red_splits<true, true>(kt + nt, cdiv(M, 64), tc.smem);
    if (!make_map(&mXmn, X, K, M, K, 64) || !make_map(&mGmn, G, R, M, R, 64) ||
        !make_map(&mdYmn, dY, N, M, N, 64) || !make_map(&mXAmn, XA_saved, R, M, R, 64))
      return QLORA_ERR_CUDA;
    GemmArgs ga = base_args(err);
    ga.M = static_cast<int32_t>(K);
    ga.N = static_cast<int32_t>(R);
    ga.mode = GM_PLAIN;
    ga.red_len = static_cast<int32_t>(M);
    ga.out_valid = static_cast<int32_t>(R);
    ga.red_scale = s;
    ga.red_f32 = dA;
    ga.red_ld = R;
    ga.red_accumulate = accumulate ? 1 : 0;
    GemmArgs gb = base_args(err);
    gb.M = static_cast<int32_t>(N);
    gb.N = r;
    gb.mode = GM_DB;
    gb.red_len = static_cast<int32_t>(M);
    gb.r = r;
    gb.nseg = n_seg;
    for (int j = 0; j <= n_seg; ++j) gb.seg_start[j] = sg.start[j];
    gb.out_valid = r;
    gb.red_scale = s;
    gb.red_f32_t = dB;
    gb.red_ld_t = N;
    gb.red_accumulate = accumulate ? 1 : 0;
    const RedProb pb{gb, mdYmn, mXAmn, nt, 1, 1, bn_b};
    QL_TRY((launch_gemm_red<true, true>("gemm_dadb", splits, tc, RedProb{ga, mXmn, mGmn, kt, 1, 1, bn_a}, &pb,
                                        st)));
  }
  return QLORA_OK;
}
}  // namespace

extern "C" {

qlora_status qlora_linear_bwd(const void* dY, const void* X, const void* XA_saved, int64_t M, const qlora_w4* W,
                              const void* A, const void* B, int32_t r, int32_t n_seg, const int64_t* seg_n, float s,
                              void* dX, float* dA, float* dB, void* ws, size_t ws_bytes, cudaStream_t st) {
  return linear_bwd(dY, X, XA_saved, M, W, A, B, r, n_seg, seg_n, s, dX, dA, dB, ws, ws_bytes, st, false);
}

qlora_status qlora_linear_bwd_accumulate(const void* dY, const void* X, const void* XA_saved, int64_t M,
                                         const qlora_w4* W, const void* A, const void* B, int32_t r, int32_t n_seg,
                                         const int64_t* seg_n, float s, void* dX, float* dA, float* dB, void* ws,
                                         size_t ws_bytes, cudaStream_t st) {
  return linear_bwd(dY, X, XA_saved, M, W, A, B, r, n_seg, seg_n, s, dX, dA, dB, ws, ws_bytes, st, true);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// XA = X A with scratch in a static device array (for callers that cannot
// allocate the workspace).  The split partial sums go through the array and
// a separate reduction kernel; the split count is the forward's (xa_splits)
// and both sum the splits in split order from zero, so the result equals
// qlora_linear_fwd's XA_save, which sums on chip.
// Array layout: a 256-byte header whose first word collects device-side
// failures (zero when the module loads, cleared by the status query), then
// A^T [R, K] bf16, then the fp32 split partials of one row chunk.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_xa_static_scratch[QLORA_XA_STATIC_SCRATCH_BYTES];

namespace {
constexpr size_t kStaticHeader = 256;
std::mutex g_xa_static_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The current CUDA context (driver entry point fetched through the runtime):
// a module -- and with it the static array -- belongs to one context, so a
// cached address is only valid for the context it was looked up in.
CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

struct StaticAddr {
  int dev;
  CUcontext ctx;
  void* addr;
};
std::vector<StaticAddr> g_xa_static_addr;

// Device address of the static array in the current device's current
// context, looked up (cudaGetSymbolAddress, with that device current) the
// first time this device and context are seen.
qlora_status xa_static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QLORA_ERR_CUDA;
  const CUcontext ctx = current_context();  // null before the runtime made one current: looked up again later
  std::lock_guard<std::mutex> lk(g_xa_static_mu);
  for (const StaticAddr& a : g_xa_static_addr)
    if (a.dev == dev && a.ctx == ctx) {
      *out = a.addr;
      return QLORA_OK;
    }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_xa_static_scratch) != cudaSuccess || !p) return QLORA_ERR_CUDA;
  g_xa_static_addr.push_back({dev, ctx, p});
  *out = p;
  return QLORA_OK;
}
}  // namespace

extern "C" qlora_status qlora_linear_xa_static(const void* X, int64_t M, int64_t K, const void* A, int32_t R,
                                               void* XA, cudaStream_t st) {
  if (!X || !A || !XA) return QLORA_ERR_INVALID_ARG;
  if (M < 0 || K < 64 || R < 8 || R > 256 || R % 8 != 0) return QLORA_ERR_INVALID_ARG;
  if (K % 64 != 0 || K > (int64_t(1) << 30) || M > (int64_t(1) << 30)) return QLORA_ERR_UNSUPPORTED;
  if (!al16(X) || !al16(A) || !al16(XA)) return QLORA_ERR_ALIGNMENT;
  const size_t cap = QLORA_XA_STATIC_SCRATCH_BYTES - kStaticHeader;
  const int splits = xa_splits(M, K, R);
  const size_t at_bytes = align256(size_t(R) * K * 2);
  const size_t per_row = size_t(splits) * R * 4;
  if (at_bytes + 128 * per_row > cap) return QLORA_ERR_WORKSPACE;
  if (M == 0) return QLORA_OK;
  int64_t rows_per_chunk = static_cast<int64_t>((cap - at_bytes) / per_row) / 128 * 128;
  rows_per_chunk = std::min<int64_t>(rows_per_chunk, rup(M, 128));
  void* base = nullptr;
  QL_TRY(xa_static_scratch(&base));
  if (!encode_fn()) return QLORA_ERR_CUDA;
  uint8_t* b8 = static_cast<uint8_t*>(base);
  uint32_t* err = reinterpret_cast<uint32_t*>(b8);
  void* At = b8 + kStaticHeader;
  float* part = reinterpret_cast<float*>(b8 + kStaticHeader + at_bytes);

  {
    const TransposeJob jobs[1] = {tjob(A, K, R, R, At, R, K, K)};
    QL_TRY(launch_transposes("transpose_A_static", jobs, 1, st));
  }
  const int bn = static_cast<int>(rup(R, 16));
  const TileCfg tc = tile_cfg(bn);
  CUtensorMap mAt;
  if (!make_map(&mAt, At, K, R, K, static_cast<uint32_t>(bn))) return QLORA_ERR_CUDA;
  for (int64_t m0 = 0; m0 < M; m0 += rows_per_chunk) {
    const int64_t mc = std::min<int64_t>(rows_per_chunk, M - m0);
    const void* Xc = static_cast<const uint8_t*>(X) + size_t(m0) * K * 2;
    CUtensorMap mX;
    if (!make_map(&mX, Xc, K, mc, K, 128)) return QLORA_ERR_CUDA;
    GemmArgs g = base_args(err);
    g.M = static_cast<int32_t>(mc);
    g.N = R;
    g.mode = GM_PLAIN;
    g.red_len = static_cast<int32_t>(K);
    g.splits = splits;
    g.out_ld = R;
    g.out_valid = R;
    g.out_split_stride = mc * R;
    g.out = part;
    QL_TRY((launch_gemm<false, false, EPI_F32_PART>("gemm_xa_static", dim3(static_cast<unsigned>(cdiv(mc, 128)), 1, splits), tc, mX,
                                     mAt, mX, mAt, g, st)));
    ReduceArgs ra = reduce_args(part, splits, mc, R, R, mc * R, 1.0f);
    ra.out_bf16 = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(XA) + size_t(m0) * R * 2);
    ra.ld_o = R;
    QL_TRY(launch_reduce("reduce_xa_static", ra, st));
  }
  return QLORA_OK;
}

extern "C" qlora_status qlora_linear_xa_static_status(cudaStream_t st) {
  void* base = nullptr;
  QL_TRY(xa_static_scratch(&base));
  if (cudaStreamSynchronize(st) != cudaSuccess) return QLORA_ERR_CUDA;
  uint32_t flag = 0;
  if (cudaMemcpy(&flag, base, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return QLORA_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return QLORA_ERR_CUDA;
  if (flag != 0) {
    if (cudaMemsetAsync(base, 0, 4, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
      return QLORA_ERR_CUDA;
    return QLORA_ERR_TIMEOUT;
  }
  return QLORA_OK;
}
