// Host side of the C ABI (include/dg.h): argument validation, the tile-size
// heuristic, TMA tensor-map encoding and the launch of the sm_103a kernels.
//
// The entry points follow DeepGEMM's interface (deepep.org/zh/deepgemm,
// "接口设计"; es.news.hada.io/topic?id=19459, "Interfaz GEMM y restricciones de
// layout", "Dense y Grouped GEMM", "Utilidades y variables de entorno").
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "dg.h"
#include "dg_instances.cuh"
#include "dg_quant.h"

// The device status word: kernels record the first device-side error here.
// One word per device, shared by every stream and call on it.
__device__ unsigned int g_dg_status = 0;
// Where take_status_kernel leaves the value it took from the status word.
__device__ unsigned int g_dg_status_taken = 0;

// Reads and clears the status word in one atomic exchange, so that an error
// raised by a kernel on another stream between the read and the clear is not
// lost (it stays in the word for the next read).
__global__ void take_status_kernel() { g_dg_status_taken = atomicExch(&g_dg_status, 0u); }

namespace {

using dgk::Instance;

thread_local std::string t_err;

dg_status fail(dg_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return s;
}

dg_status ok() {
  t_err.clear();
  return DG_OK;
}

std::atomic<int> g_num_sms_limit{0};
std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<int> g_skip_producer{0};
std::atomic<int> g_force_bn{-1};     // -1: not read from the environment yet; 0: auto
std::atomic<int> g_force_split{0};
std::atomic<int> g_force_pair{-1};   // -1: heuristic; 0: no pair form; 1: pair form only
std::atomic<int> g_force_bs{-1};     // -1: heuristic; 0: no block-scaled kernel; 1: only those

constexpr int kMaxSmem = 232448;     // 227 KB per CTA on sm_100-class GPUs
constexpr int kMaxDevices = 64;
constexpr int kMaxCluster = 8;
constexpr int kRasterM = 16;
constexpr int kMaxInstances = 32;    // instances per table (the cluster cache's size)

void read_env_once() {
  int expected = -1;
  if (!g_force_bn.compare_exchange_strong(expected, 0)) return;
  // DG_FORCE_PAIR=0|1 (tests and benchmarks only): as dg_debug_force_pair
  if (const char* s = std::getenv("DG_FORCE_PAIR")) g_force_pair.store(std::atoi(s) ? 1 : 0);
  // DG_FORCE_BLOCK_SCALED=0|1 (tests and benchmarks only): as dg_debug_force_block_scaled
  if (const char* s = std::getenv("DG_FORCE_BLOCK_SCALED"))
    g_force_bs.store(std::atoi(s) ? 1 : 0);
  // DG_FORCE_CONFIG="block_n,split_k" (tests and benchmarks only)
  if (const char* s = std::getenv("DG_FORCE_CONFIG")) {
    int bn = 0, sp = 0;
    if (std::sscanf(s, "%d,%d", &bn, &sp) >= 1) {
      g_force_bn.store(bn);
      g_force_split.store(sp);
    }
  }
}

bool print_configs() {
  const char* s = std::getenv("DG_PRINT_CONFIGS");
  return s && s[0] && s[0] != '0';
}

// ------------------------------------------------------------ instances --
struct Table {
  const Instance* p;
  int n;
};

// Instance tables: 0 dense nt, 1 contiguous, 2 masked, 3 MN-major operands
// (dense nn / tn / tt and the K-grouped form); 4-7 the same with packed UE8M0
// scales: the block-scaled instances first, then those that decode the scales
// into the promotion (which also hold the K-split forms).
constexpr int kNumTables = 8;

// Block-scaled and promotion instances of one packed-UE8M0 table, concatenated
// once (thread-safe static initialisation).
template <const dgk::Instance* (*BS)(int*), const dgk::Instance* (*SFP)(int*)>
Table joined() {
  static const std::vector<Instance> all = [] {
    int nb = 0, ns = 0;
    const Instance* b = BS(&nb);
    const Instance* f = SFP(&ns);
    std::vector<Instance> v(b, b + nb);
    v.insert(v.end(), f, f + ns);
    return v;
  }();
  return Table{all.data(), static_cast<int>(all.size())};
}

int table_id(int kind, int layout, bool sfp = false) {
  return ((layout != dgk::kNT || kind == dgk::kKGrouped) ? 3 : kind) + (sfp ? 4 : 0);
}

Table table_for(int tid) {
  Table t{nullptr, 0};
  switch (tid) {
    case 0: t.p = dgk::instances_dense(&t.n); break;
    case 1: t.p = dgk::instances_contiguous(&t.n); break;
    case 2: t.p = dgk::instances_masked(&t.n); break;
    case 3: t.p = dgk::instances_mn(&t.n); break;
    case 4: t = joined<dgk::instances_bs_dense, dgk::instances_dense_ue8m0>(); break;
    case 5: t = joined<dgk::instances_bs_contiguous, dgk::instances_contiguous_ue8m0>(); break;
    case 6: t = joined<dgk::instances_bs_masked, dgk::instances_masked_ue8m0>(); break;
    default: t = joined<dgk::instances_bs_mn, dgk::instances_mn_ue8m0>(); break;
  }
  return t;
}

int smem_for(const Instance& in, int kb, int num_groups) {
  // the promotion kernels keep two tiles' B scales in shared memory (one
  // buffer filled while the other is read); the block-scaled ones read them
  // into the scale-factor staging instead
  int s = in.fixed_smem + (in.bs ? 0 : 2 * dgk::sb_buf_words(kb) * 4) +
          (in.mode == dgk::kMasked     ? (2 * num_groups + 1) * 4
           : in.mode == dgk::kKGrouped ? (num_groups + 1) * 4
                                       : 0);
  return (s + 15) & ~15;
}

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// ------------------------------------------------------------ heuristic --
// A plan: one instance, the K split (cluster size) and the persistent grid.
struct Plan {
  int inst = -1;
  int split = 1;
  int pair = 0;
  long long tiles = 0;
  int clusters = 0;
  int smem = 0;
};

// Estimated kernel time (us) of one configuration.  The constants are fitted
// to timings of every configuration of the dense decode and prefill sweeps on
// GB300 (median error ~8%):
//  * a CTA's K group costs the slowest of: the MMA/promotion cadence (0.22 us
//    for 128-wide tiles, 0.50 us for 256-wide, 0.39 us for a CTA pair's
//    256 x 256 tile), its share of HBM bandwidth for the B tile (~9 TB/s
//    aggregate, L2 hits included; a B tile is read from DRAM once by the M
//    blocks of a raster band that share it), and the SM's TMA ingest for A
//    and B (~100 GB/s per SM);
//  * each wave of CTAs pays ~3 us before its first operands land and a tail
//    (~4.9 us for the K split's cluster reduction, ~1.6 us otherwise);
//  * a persistent CTA pays ~0.9 us per extra tile (epilogue), plus ~1.9 us per
//    launch.
// A split whose clusters do not all fit at once runs in several waves, each
// paying its own head and tail: this is what the model must steer away from.
double est_time_us(const Instance& in, int S, long long tiles, long long clusters_resident,
                   int num_sms, int kind, long long m_rows, int n, int k, int num_groups) {
  (void)n;
  // block-scaled: ~0.39 us per K group and CTA at 256 columns, 0.38 at 224
  // (two accumulators), 0.375 at 128, 0.41 per K group of a CTA pair (fitted
  // to every width on the prefill, contiguous and masked sweeps: the TMA
  // writes and the MMAs' operand reads share the SM's shared-memory
  // bandwidth); the MMA alone would take 0.13-0.27 us
  // (the promotion kernels' packed-scale twins: ~18% slower per K group than
  // with fp32 scales, measured on the prefill shapes)
  const double t_cad = in.bs ? (in.pair ? 0.41
                                        : in.block_n <= 128 ? 0.375 : in.block_n == 224 ? 0.38 : 0.387)
                             : (in.pair ? 0.39 : (in.block_n <= 128 ? 0.22 : 0.50)) *
                                   (in.sfp ? 1.18 : 1.0);
  const double bw_hbm = 9.0e6;   // bytes / us, whole GPU
  const double bw_sm = 102e3;    // bytes / us, one SM's TMA ingest
  // the K split's reduction moves BN columns of fp32 partials per row: its
  // tail grows with the tile width (fit to the decode sweep: 64-wide tiles
  // split 4 ways 10.7 us against 12.3-13.4 for 128-wide on 128x2112x7168)
  const double head = 3.06, tail = S > 1 ? 1.6 + 3.3 * in.block_n / 128.0 : 1.6, fixed = 1.9;
  // (fitted: a block-scaled kernel with one accumulator waits for each
  // tile's epilogue, ~0.9 us more per tile, with two ~0.2 us; the promotion
  // kernels' packed-scale twins decode the scales of every K group, which
  // weighs on short-K tiles)
  const double per_tile = 0.92 + (in.bs ? (in.nacc == 1 ? 0.9 : 0.18) : 0.0) +
                          (!in.bs && in.sfp ? 0.7 : 0.0);
  const long long kb = k / 128;
  const long long kper = cdiv(kb, S);
  // the A box the TMA fills per K group (rows past M are zero-filled, not free)
  const double a_rows = in.a_rows;
  const double b_rows = in.pair ? in.block_n / 2.0 : (double)in.block_n;
  long long ctas, waves = 1, groups, ntile = 1;
  if (in.split) {
    const long long cl = std::max<long long>(1, std::min(tiles, clusters_resident));
    waves = cdiv(tiles, std::max<long long>(1, clusters_resident));
    ctas = cl * S;
    groups = kper;
  } else if (in.pair) {
    const long long pairs = std::max<long long>(1, std::min(tiles, clusters_resident));
    ctas = 2 * pairs;
    ntile = cdiv(tiles, pairs);
    groups = ntile * kb;
  } else {
    ctas = std::max<long long>(1, std::min<long long>(tiles, num_sms));
    ntile = cdiv(tiles, ctas);
    groups = ntile * kb;
  }
  // B tiles come from DRAM once per raster band of M blocks that share them
  // (dense; the M blocks of one expert in the contiguous form).  The masked
  // form's few M blocks per group are taken as reading theirs each (fitted:
  // the masked sweep's choices).
  const long long bm = in.pair ? 256 : 128;
  long long reuse = kind == dgk::kContiguous ? cdiv(m_rows, bm) / std::max(1, num_groups)
                    : kind == dgk::kMasked   ? 1
                                             : cdiv(m_rows, bm);
  reuse = std::max(1LL, std::min<long long>(reuse, kRasterM));
  const double t_mem = b_rows * 128.0 / (double)reuse / (bw_hbm / (double)ctas);
  const double t_tma = in.bs ? 0.0 : (a_rows + b_rows) * 128.0 / bw_sm;
  const double tg = std::max(t_cad, std::max(t_mem, t_tma));
  return fixed + (double)waves * (head + (double)groups * tg + tail) + (double)(ntile - 1) * per_tile;
}

bool has_split64(const Table& tab) {
  for (int i = 0; i < tab.n; ++i)
    if (tab.p[i].split && tab.p[i].a_rows == 64) return true;
  return false;
}

// cap(S): clusters of S CTAs that can be resident at once.
// K-grouped form: k is the whole K (the operands' rows); the model takes each
// tile as an average group's K, k / num_groups.
template <typename Cap>
Plan choose(int kind, long long m_rows, int n, int k, int num_groups, int num_sms, Cap cap,
            int force_bn, int force_split, int layout = dgk::kNT, bool sfp = false) {
  const Table tab = table_for(table_id(kind, layout, sfp));
  const int kb = k / 128;
  const int k_model = kind == dgk::kKGrouped ? std::max(128, (k / std::max(1, num_groups)) / 128 * 128) : k;
  Plan best;
  double best_cost = 1e300;
  for (int i = 0; i < tab.n; ++i) {
    const Instance& in = tab.p[i];
    if (in.mode != kind || in.layout != layout) continue;
    if (force_bn > 0 && in.block_n != force_bn) continue;
    // 64-row A tiles serve M <= 64 only.  Timed alone (cold L2) they matched
    // the full-A split, but in the back-to-back decode sweep the sweep took
    // 186.4 us with them and 168.2 us without, so the heuristic takes them
    // only under a forced configuration (where they remain the M <= 64 choice).
    const bool forced = force_bn > 0 || force_split > 0;
    if (in.a_rows < 128 && (m_rows > in.a_rows || !forced)) continue;
    // The CTA-pair form measured slower than the 128-row form on every shape
    // so far (the promotion kernels: their promotion, not the MMA, sets the
    // pace; the block-scaled ones: 1-15% on the prefill shapes, up to 1.7x on
    // the masked ones): it runs only when forced.
    const int fp = g_force_pair.load();
    if (fp == 0 && in.pair) continue;
    if (fp < 0 && in.pair) continue;
    if (fp == 1 && !in.pair) continue;
    const int fbs = g_force_bs.load();
    if ((fbs == 0 && in.bs) || (fbs == 1 && !in.bs)) continue;
    if (forced && in.a_rows == 128 && in.split && m_rows <= 64 && has_split64(tab)) continue;
    const int smem = smem_for(in, kb, num_groups);
    if (smem > kMaxSmem) continue;
    // the K split is for shapes whose output tiles cannot fill the SMs
    if (in.split && force_split == 0 &&
        (kind == dgk::kMasked ? (long long)num_groups * cdiv(m_rows, 128) : cdiv(m_rows, 128)) *
                cdiv(n, in.block_n) >= num_sms)
      continue;
    const int s_lo = in.split ? 2 : 1;
    // the heuristic splits no finer than one K group per CTA; a forced split
    // may (the CTAs without a K group add zeros)
    const int s_hi = in.split ? (force_split > 0 ? kMaxCluster : std::min(kMaxCluster, kb)) : 1;
    for (int S = s_lo; S <= s_hi; ++S) {
      if (force_split > 0 && S != force_split) continue;
      if (force_split == 0 && force_bn > 0 && in.split) {
        // a forced block_n without a forced split keeps the unsplit instance
        continue;
      }
      long long mblk;
      if (kind == dgk::kMasked || kind == dgk::kKGrouped)
        mblk = (long long)num_groups * cdiv(m_rows, in.pair ? 256 : 128);
      else mblk = cdiv(m_rows, in.pair ? 256 : 128);
      const long long tiles = mblk * cdiv(n, in.block_n);
      const long long c = std::max(1, cap(i, in, in.pair ? 2 : S, smem));
      const double t = est_time_us(in, S, tiles, c, num_sms, kind, m_rows, n, k_model, num_groups);
      const double cost = t;
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best.inst = i;
        best.split = S;
        best.tiles = tiles;
        // the split form runs one cluster per tile (its epilogue reuses the
        // operand ring); the others are persistent, at most one wave of CTAs
        best.clusters = in.split ? (int)tiles : (int)std::min<long long>(tiles, c);
        best.pair = in.pair;
        best.smem = smem;
      }
    }
  }
  return best;
}

}  // namespace

namespace {

// ------------------------------------------------------- device state ----
struct DeviceState {
  bool ready = false;
  int sms = 0;
  unsigned int* status = nullptr;
  // resident clusters per (instance table, instance, split)
  int max_clusters[kNumTables][kMaxInstances][kMaxCluster + 1] = {};
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

dg_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Set-up of the current device, once: architecture check, the status word's
// address, the tensor-map encoder, and the shared-memory limit of every
// instance.
dg_status device_state(DeviceState** out, int* dev_out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DG_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
  }
  if (dev < 0 || dev >= kMaxDevices) return fail(DG_ERR_NO_DEVICE, "device index %d", dev);
  DeviceState& st = g_dev[dev];
  *dev_out = dev;
  std::lock_guard<std::mutex> lock(g_mu);
  if (st.ready) {
    *out = &st;
    return DG_OK;
  }
  int major = 0, minor = 0, sms = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(DG_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a", dev, major,
                minor);
  void* sp = nullptr;
  if ((e = cudaGetSymbolAddress(&sp, g_dg_status)) != cudaSuccess)
    return cuda_fail(e, "cudaGetSymbolAddress(status)");
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return fail(DG_ERR_CUDA, "cuTensorMapEncodeTiled not available");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  for (int tid = 0; tid < kNumTables; ++tid) {
    const Table tab = table_for(tid);
    if (tab.n > kMaxInstances)
      return fail(DG_ERR_CUDA, "instance table %d holds %d instances, more than %d", tid, tab.n,
                  kMaxInstances);
    for (int i = 0; i < tab.n; ++i)
      if ((e = tab.p[i].set_smem(kMaxSmem)) != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
  }
  st.sms = sms;
  st.status = static_cast<unsigned int*>(sp);
  st.ready = true;
  *out = &st;
  return DG_OK;
}

int clusters_resident(DeviceState& st, int kind, int inst, const Instance& in, int S, int smem,
                      int num_sms) {
  if (S <= 1) return num_sms;
  if (inst < 0 || inst >= kMaxInstances || S > kMaxCluster) return 0;
  // the cache is filled lazily by whichever thread plans first
  std::lock_guard<std::mutex> lock(g_mu);
  int& slot = st.max_clusters[table_id(kind, in.layout, in.sfp != 0)][inst][S];
  if (slot == 0) {
    int n = 0;
    if (in.max_clusters(S, kMaxSmem, &n) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = -1;
    }
    slot = n;
  }
  (void)smem;
  if (slot < 0) return 0;
  // a limit on SMs caps the clusters too
  return std::min(slot, std::max(1, num_sms / S));
}

int sms_in_use(const DeviceState& st) {
  const int lim = g_num_sms_limit.load();
  return (lim > 0 && lim < st.sms) ? lim : st.sms;
}

// ------------------------------------------------------------ tensor maps --
dg_status encode(CUtensorMap* m, CUtensorMapDataType dt, void* ptr, const uint64_t dims[3],
                 const uint64_t strides[2], const uint32_t box[3], CUtensorMapSwizzle sw,
                 CUtensorMapL2promotion l2, const char* name) {
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, dt, 3, ptr, reinterpret_cast<const cuuint64_t*>(dims),
                        reinterpret_cast<const cuuint64_t*>(strides),
                        reinterpret_cast<const cuuint32_t*>(box), estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(DG_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", name, (int)r);
  return DG_OK;
}

// A [z][rows][K] e4m3 (layout bit 0: [K][rows]), B [g][N][K] e4m3 (layout
// bit 1: [K][N]), sa [z][kb][ld_sa] fp32, D and C [zD][rows][N] bf16 (zD = zA
// unless given).  MN-major operands are read in boxes of 128 x 128 K rows.
dg_status make_maps(dgk::Maps* mp, const void* A, const float* sa, int ld_sa, const void* B,
                    void* D, int rows, int zA, int N, int K, int gB, int block_n, int a_rows,
                    const void* C = nullptr, int layout = dgk::kNT, int zD = 0,
                    bool sf_packed = false) {
  const int kb = K / 128;
  if (zD <= 0) zD = zA;
  {
    const bool mn = (layout & 1) != 0;
    const uint64_t dims[3] = {mn ? (uint64_t)rows : (uint64_t)K, mn ? (uint64_t)K : (uint64_t)rows,
                              (uint64_t)zA};
    const uint64_t str[2] = {mn ? (uint64_t)rows : (uint64_t)K, (uint64_t)rows * K};
    const uint32_t box[3] = {128, mn ? 128u : (uint32_t)a_rows, 1};
    dg_status s = encode(&mp->a, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void*>(A), dims, str,
                         box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "A");
    if (s != DG_OK) return s;
  }
  {
    const bool mn = (layout & 2) != 0;
    const uint64_t dims[3] = {mn ? (uint64_t)N : (uint64_t)K, mn ? (uint64_t)K : (uint64_t)N,
                              (uint64_t)gB};
    const uint64_t str[2] = {mn ? (uint64_t)N : (uint64_t)K, (uint64_t)N * K};
    const uint32_t box[3] = {128, mn ? 128u : (uint32_t)block_n, 1};
    dg_status s = encode(&mp->b, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void*>(B), dims, str,
                         box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "B");
    if (s != DG_OK) return s;
  }
  if (sf_packed) {
    // packed UE8M0 words [z][ceil(kb/4)][ld_sa]: two words per ring slot
    const int kbp = (kb + 3) / 4;
    const uint64_t dims[3] = {(uint64_t)ld_sa, (uint64_t)kbp, (uint64_t)zA};
    const uint64_t str[2] = {(uint64_t)ld_sa * 4, (uint64_t)kbp * ld_sa * 4};
    const uint32_t box[3] = {128, 2, 1};
    dg_status s = encode(&mp->sa, CU_TENSOR_MAP_DATA_TYPE_INT32, const_cast<float*>(sa), dims,
                         str, box, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         "sfa");
    if (s != DG_OK) return s;
  } else {
    const uint64_t dims[3] = {(uint64_t)ld_sa, (uint64_t)kb, (uint64_t)zA};
    const uint64_t str[2] = {(uint64_t)ld_sa * 4, (uint64_t)kb * ld_sa * 4};
    const uint32_t box[3] = {128, (uint32_t)dgk::SA_GROUPS, 1};
    dg_status s = encode(&mp->sa, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, const_cast<float*>(sa), dims,
                         str, box, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         "sa");
    if (s != DG_OK) return s;
  }
  {
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)rows, (uint64_t)zD};
    const uint64_t str[2] = {(uint64_t)N * 2, (uint64_t)rows * N * 2};
    const uint32_t box[3] = {32, 128, 1};
    dg_status s = encode(&mp->d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, "D");
    if (s != DG_OK) return s;
    // the addend C: loaded into the staging tile in exactly the store's layout
    if (C) {
      s = encode(&mp->c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(C), dims, str, box,
                 CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "C");
      if (s != DG_OK) return s;
    } else {
      std::memset(&mp->c, 0, sizeof(mp->c));
    }
  }
  return DG_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace {

const char* kind_name(int kind) {
  return kind == dgk::kDense        ? "dense"
         : kind == dgk::kContiguous ? "contiguous"
         : kind == dgk::kMasked     ? "masked"
                                    : "k-grouped";
}

const char* layout_name(int layout) {
  return layout == dgk::kNT ? "nt" : layout == dgk::kNN ? "nn" : layout == dgk::kTN ? "tn" : "tt";
}

// Shared path of the GEMM entry points.  rows = M (dense, K-grouped), M_total
// (contiguous) or max_m (masked); idx = m_indices, masked_m or ks; K = the
// whole K (K-grouped: the operands' rows, all groups together).
dg_status run(int kind, const void* A, const float* sa, int ld_sa, const void* B, const float* sb,
              void* D, const int32_t* idx, int rows, int N, int K, int G, int expected_m,
              void* stream, const void* C = nullptr, int layout = dgk::kNT,
              bool sf_packed = false) {
  read_env_once();
  // -------- validation (host only; nothing is launched on an error) ------
  if (rows < 0 || N < 0 || K < 0)
    return fail(DG_ERR_INVALID_ARG, "negative size (rows=%d, N=%d, K=%d)", rows, N, K);
  const int max_groups = kind == dgk::kMasked     ? dgk::MAX_GROUPS_MASKED
                         : kind == dgk::kKGrouped ? dgk::MAX_GROUPS_KGROUPED
                                                  : 0x7fffffff;
  if (kind != dgk::kDense && (G < 1 || G > max_groups))
    return fail(DG_ERR_INVALID_ARG, "num_groups=%d outside [1, %d]", G, max_groups);
  if ((layout & 1) && rows % 16 != 0)
    return fail(DG_ERR_UNSUPPORTED_SHAPE, "M=%d: A stored [K][M] needs M a multiple of 16", rows);
  if (K % 128 != 0 || K < 128 || K > 128 * dgk::MAX_KB)
    return fail(DG_ERR_UNSUPPORTED_SHAPE, "K=%d: need a multiple of 128 in [128, %d]", K,
                128 * dgk::MAX_KB);
  if (N % 16 != 0 || N < 16)
    return fail(DG_ERR_UNSUPPORTED_SHAPE, "N=%d: need a multiple of 16, at least 16", N);
  if (kind == dgk::kContiguous && rows % 128 != 0)
    return fail(DG_ERR_UNSUPPORTED_SHAPE, "M_total=%d is not a multiple of 128", rows);
  if (!A || !sa || !B || !sb || !D)
    return fail(DG_ERR_INVALID_ARG, "null tensor pointer");
  if (kind != dgk::kDense && !idx)
    return fail(DG_ERR_INVALID_ARG, "null %s",
                kind == dgk::kMasked ? "masked_m" : kind == dgk::kKGrouped ? "ks" : "m_indices");
  if (!aligned16(A) || !aligned16(B) || !aligned16(D) || !aligned16(sa) || (C && !aligned16(C)) ||
      (reinterpret_cast<uintptr_t>(sb) & 3u) || (idx && (reinterpret_cast<uintptr_t>(idx) & 3u)))
    return fail(DG_ERR_MISALIGNED, "A, B, C, D and sa need 16-byte alignment, sb and indices 4");
  if (ld_sa < rows || ld_sa % 4 != 0 || ld_sa < 1)
    return fail(ld_sa % 4 != 0 ? DG_ERR_MISALIGNED : DG_ERR_INVALID_ARG,
                "ld_sa=%d: need >= %d and a multiple of 4", ld_sa, rows);
  if ((long long)rows * (long long)G >= (1ll << 31) || (long long)N * K >= (1ll << 40))
    return fail(DG_ERR_UNSUPPORTED_SHAPE, "tensor too large");
  if (rows == 0) return ok();  // nothing to compute

  // -------- device, plan, tensor maps, launch ------------------------------
  DeviceState* st = nullptr;
  int dev = 0;
  dg_status s = device_state(&st, &dev);
  if (s != DG_OK) return s;
  const int num_sms = sms_in_use(*st);
  auto cap = [&](int i, const Instance& in, int S, int smem) {
    return S <= 1 ? num_sms : clusters_resident(*st, kind, i, in, S, smem, num_sms);
  };
  const int m_plan = kind == dgk::kMasked ? std::max(1, std::min(expected_m, rows)) : rows;
  const Plan pl = choose(kind, m_plan, N, K, G, num_sms, cap, g_force_bn.load(),
                         g_force_split.load(), layout, sf_packed);
  if (pl.inst < 0)
    return fail(DG_ERR_UNSUPPORTED_SHAPE, "no kernel configuration for this shape%s",
                g_force_bn.load() > 0 ? " (DG_FORCE_CONFIG)" : "");
  const Instance& in = table_for(table_id(kind, layout, sf_packed)).p[pl.inst];
  int clusters = pl.clusters;
  if (kind == dgk::kMasked) {
    // the device decides how many tiles there are: launch for the most that can
    // exist, at most one resident wave of CTAs (pairs: of 2-CTA clusters)
    const long long ub = (long long)G * cdiv(rows, in.pair ? 256 : 128) * cdiv(N, in.block_n);
    const int resident = in.pair ? std::max(1, cap(pl.inst, in, 2, pl.smem)) : num_sms;
    clusters = (int)std::min<long long>(ub, resident);
  }
  const int grid = std::max(1, clusters) * (in.pair ? 2 : pl.split);

  dgk::Maps maps;
  const bool has_c = kind == dgk::kDense || kind == dgk::kKGrouped;
  // rows of B per TMA box: the tile, or half of it per CTA of a pair
  const int b_box = in.pair ? in.block_n / 2 : in.block_n;
  s = make_maps(&maps, A, sa, ld_sa, B, D, rows, kind == dgk::kMasked ? G : 1, N, K,
                (kind == dgk::kDense || kind == dgk::kKGrouped) ? 1 : G, b_box, in.a_rows,
                has_c ? C : nullptr, layout, kind == dgk::kKGrouped ? G : 0, sf_packed);
  if (s != DG_OK) return s;

  dgk::Params p{};
  p.M = rows;
  p.N = N;
  p.K = K;
  p.kb = K / 128;
  p.nb = (N + 127) / 128;
  p.num_groups = kind == dgk::kDense ? 1 : G;
  p.ks = kind == dgk::kKGrouped ? idx : nullptr;
  p.num_m_blocks = (int)cdiv(rows, in.pair ? 256 : 128);
  p.num_n_blocks = (int)cdiv(N, in.block_n);
  p.raster_m = kRasterM;
  p.split_k = pl.split;
  p.sb = sb;
  p.kbp = (K / 128 + 3) / 4;
  p.sa_packed = sf_packed ? static_cast<const void*>(sa) : nullptr;
  p.ld_sa = ld_sa;
  p.m_indices = kind == dgk::kContiguous ? idx : nullptr;
  p.masked_m = kind == dgk::kMasked ? idx : nullptr;
  p.D = static_cast<uint16_t*>(D);
  p.C = has_c ? static_cast<const uint16_t*>(C) : nullptr;
  p.status = st->status;
  p.timeout_ns = g_timeout_ns.load();
  p.debug_flags = g_skip_producer.load() ? dgk::DBG_SKIP_PRODUCER : 0u;

  const cudaError_t e = in.launch(maps, p, grid, in.pair ? 2 : pl.split, pl.smem,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "kernel launch");
  }
  if (print_configs())
    std::fprintf(stderr,
                 "[dg] %s %s%s M=%d N=%d K=%d G=%d: block_n=%d split_k=%d pair=%d stages=%d "
                 "tiles=%lld grid=%d smem=%d%s\n",
                 kind_name(kind), layout_name(layout), sf_packed ? " ue8m0" : "", rows, N, K, G,
                 in.block_n, pl.split, in.pair, in.stages, (long long)pl.tiles, grid, pl.smem,
                 in.bs ? " block-scaled" : "");
  return ok();
}

}  // namespace

// ====================================================================== ABI ==
extern "C" {

dg_status dg_gemm_fp8_fp8_bf16_nt(const void* A, const float* sa, int ld_sa, const void* B,
                                  const float* sb, void* D, int M, int N, int K, void* stream) {
  return run(dgk::kDense, A, sa, ld_sa, B, sb, D, nullptr, M, N, K, 1, M, stream);
}

dg_status dg_gemm_fp8_fp8_bf16_nt_add_c(const void* A, const float* sa, int ld_sa, const void* B,
                                        const float* sb, const void* C, void* D, int M, int N,
                                        int K, void* stream) {
  if (!C) return fail(DG_ERR_INVALID_ARG, "null addend C (use dg_gemm_fp8_fp8_bf16_nt)");
  return run(dgk::kDense, A, sa, ld_sa, B, sb, D, nullptr, M, N, K, 1, M, stream, C);
}

dg_status dg_gemm_fp8_fp8_bf16_nn(const void* A, const float* sa, int ld_sa, const void* B,
                                  const float* sb, const void* C, void* D, int M, int N, int K,
                                  void* stream) {
  return run(dgk::kDense, A, sa, ld_sa, B, sb, D, nullptr, M, N, K, 1, M, stream, C, dgk::kNN);
}

dg_status dg_gemm_fp8_fp8_bf16_tn(const void* A, const float* sa, int ld_sa, const void* B,
                                  const float* sb, const void* C, void* D, int M, int N, int K,
                                  void* stream) {
  return run(dgk::kDense, A, sa, ld_sa, B, sb, D, nullptr, M, N, K, 1, M, stream, C, dgk::kTN);
}

dg_status dg_gemm_fp8_fp8_bf16_tt(const void* A, const float* sa, int ld_sa, const void* B,
                                  const float* sb, const void* C, void* D, int M, int N, int K,
                                  void* stream) {
  return run(dgk::kDense, A, sa, ld_sa, B, sb, D, nullptr, M, N, K, 1, M, stream, C, dgk::kTT);
}

dg_status dg_k_grouped_gemm_fp8_fp8_bf16_tn_contiguous(const void* A, const float* sa, int ld_sa,
                                                       const void* B, const float* sb,
                                                       const void* C, void* D, const int32_t* ks,
                                                       int num_groups, int M, int N, int K_total,
                                                       void* stream) {
  return run(dgk::kKGrouped, A, sa, ld_sa, B, sb, D, ks, M, N, K_total, num_groups, M, stream, C,
             dgk::kTN);
}

dg_status dg_gemm_fp8_fp8_bf16_nt_ue8m0(const void* A, const int32_t* sfa, int ld_sfa,
                                        const void* B, const int32_t* sfb, void* D, int M, int N,
                                        int K, void* stream) {
  return run(dgk::kDense, A, reinterpret_cast<const float*>(sfa), ld_sfa, B,
             reinterpret_cast<const float*>(sfb), D, nullptr, M, N, K, 1, M, stream, nullptr,
             dgk::kNT, true);
}

dg_status dg_gemm_fp8_fp8_bf16_nn_ue8m0(const void* A, const int32_t* sfa, int ld_sfa,
                                        const void* B, const int32_t* sfb, const void* C, void* D,
                                        int M, int N, int K, void* stream) {
  return run(dgk::kDense, A, reinterpret_cast<const float*>(sfa), ld_sfa, B,
             reinterpret_cast<const float*>(sfb), D, nullptr, M, N, K, 1, M, stream, C, dgk::kNN,
             true);
}

dg_status dg_gemm_fp8_fp8_bf16_tn_ue8m0(const void* A, const int32_t* sfa, int ld_sfa,
                                        const void* B, const int32_t* sfb, const void* C, void* D,
                                        int M, int N, int K, void* stream) {
  return run(dgk::kDense, A, reinterpret_cast<const float*>(sfa), ld_sfa, B,
             reinterpret_cast<const float*>(sfb), D, nullptr, M, N, K, 1, M, stream, C, dgk::kTN,
             true);
}

dg_status dg_gemm_fp8_fp8_bf16_tt_ue8m0(const void* A, const int32_t* sfa, int ld_sfa,
                                        const void* B, const int32_t* sfb, const void* C, void* D,
                                        int M, int N, int K, void* stream) {
  return run(dgk::kDense, A, reinterpret_cast<const float*>(sfa), ld_sfa, B,
             reinterpret_cast<const float*>(sfb), D, nullptr, M, N, K, 1, M, stream, C, dgk::kTT,
             true);
}

dg_status dg_k_grouped_gemm_fp8_fp8_bf16_tn_contiguous_ue8m0(
    const void* A, const int32_t* sfa, int ld_sfa, const void* B, const int32_t* sfb,
    const void* C, void* D, const int32_t* ks, int num_groups, int M, int N, int K_total,
    void* stream) {
  return run(dgk::kKGrouped, A, reinterpret_cast<const float*>(sfa), ld_sfa, B,
             reinterpret_cast<const float*>(sfb), D, ks, M, N, K_total, num_groups, M, stream, C,
             dgk::kTN, true);
}

dg_status dg_m_grouped_gemm_fp8_fp8_bf16_nt_contiguous_ue8m0(
    const void* A, const int32_t* sfa, int ld_sfa, const void* B, const int32_t* sfb, void* D,
    const int32_t* m_indices, int M_total, int N, int K, int num_groups, void* stream) {
  return run(dgk::kContiguous, A, reinterpret_cast<const float*>(sfa), ld_sfa, B,
             reinterpret_cast<const float*>(sfb), D, m_indices, M_total, N, K, num_groups,
             M_total, stream, nullptr, dgk::kNT, true);
}

dg_status dg_m_grouped_gemm_fp8_fp8_bf16_nt_masked_ue8m0(
    const void* A, const int32_t* sfa, int ld_sfa, const void* B, const int32_t* sfb, void* D,
    const int32_t* masked_m, int num_groups, int max_m, int N, int K, int expected_m,
    void* stream) {
  return run(dgk::kMasked, A, reinterpret_cast<const float*>(sfa), ld_sfa, B,
             reinterpret_cast<const float*>(sfb), D, masked_m, max_m, N, K, num_groups,
             expected_m, stream, nullptr, dgk::kNT, true);
}

dg_status dg_m_grouped_gemm_fp8_fp8_bf16_nt_contiguous(const void* A, const float* sa, int ld_sa,
                                                       const void* B, const float* sb, void* D,
                                                       const int32_t* m_indices, int M_total,
                                                       int N, int K, int num_groups,
                                                       void* stream) {
  return run(dgk::kContiguous, A, sa, ld_sa, B, sb, D, m_indices, M_total, N, K, num_groups,
             M_total, stream);
}

dg_status dg_m_grouped_gemm_fp8_fp8_bf16_nt_masked(const void* A, const float* sa, int ld_sa,
                                                   const void* B, const float* sb, void* D,
                                                   const int32_t* masked_m, int num_groups,
                                                   int max_m, int N, int K, int expected_m,
                                                   void* stream) {
  return run(dgk::kMasked, A, sa, ld_sa, B, sb, D, masked_m, max_m, N, K, num_groups, expected_m,
             stream);
}

namespace {
dg_status quantize(const void* X, void* Q, float* sa, int num_groups, int M, int K, int ld_sa,
                   void* stream, bool ue8m0) {
  read_env_once();
  if (!X || !Q || !sa) return fail(DG_ERR_INVALID_ARG, "dg_quantize_fp8_1x128: null pointer");
  if (num_groups < 1 || M < 0 || ld_sa < M)
    return fail(DG_ERR_INVALID_ARG, "dg_quantize_fp8_1x128: G=%d M=%d ld_sa=%d", num_groups, M,
                ld_sa);
  if (K < 128 || K % 128 != 0)
    return fail(DG_ERR_UNSUPPORTED_SHAPE, "dg_quantize_fp8_1x128: K=%d (a positive multiple of 128)",
                K);
  if ((long long)num_groups * M * (K / 128) >= (1LL << 31) || K / 128 > 65535 ||
      num_groups > 65535)
    return fail(DG_ERR_UNSUPPORTED_SHAPE,
                "dg_quantize_fp8_1x128: needs num_groups * M * K/128 < 2^31, K/128 and "
                "num_groups <= 65535");
  if (ld_sa % 4 != 0 || !aligned16(X) || !aligned16(Q) || !aligned16(sa))
    return fail(DG_ERR_MISALIGNED,
                "dg_quantize_fp8_1x128: ld_sa a multiple of 4; X, Q, sa 16-byte aligned");
  if (M == 0) return ok();  // nothing to do
  DeviceState* st = nullptr;
  int dev = 0;
  dg_status s = device_state(&st, &dev);
  if (s != DG_OK) return s;
  const cudaError_t e = dgk::launch_quantize_1x128(X, Q, sa, num_groups, M, K, ld_sa,
                                                   sms_in_use(*st),
                                                   static_cast<cudaStream_t>(stream), ue8m0);
  if (e != cudaSuccess) return cuda_fail(e, "quantiser launch");
  return ok();
}
}  // namespace

dg_status dg_quantize_fp8_1x128(const void* X, void* Q, float* sa, int num_groups, int M, int K,
                                int ld_sa, void* stream) {
  return quantize(X, Q, sa, num_groups, M, K, ld_sa, stream, false);
}

dg_status dg_quantize_fp8_1x128_ue8m0(const void* X, void* Q, int32_t* sfa, int num_groups,
                                      int M, int K, int ld_sfa, void* stream) {
  return quantize(X, Q, reinterpret_cast<float*>(sfa), num_groups, M, K, ld_sfa, stream, true);
}

int dg_get_num_sms(void) {
  const int lim = g_num_sms_limit.load();
  if (lim > 0) return lim;
  int dev = -1, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return sms;
}

dg_status dg_set_num_sms(int num_sms) {
  if (num_sms < 0) return fail(DG_ERR_INVALID_ARG, "num_sms=%d < 0", num_sms);
  int dev = -1, sms = 0;
  if (num_sms > 0 && cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      num_sms > sms)
    return fail(DG_ERR_INVALID_ARG, "num_sms=%d exceeds the device's %d SMs", num_sms, sms);
  cudaGetLastError();
  g_num_sms_limit.store(num_sms);
  return ok();
}

int dg_get_tma_aligned_size(int mn, int elem_bytes) {
  if (mn < 0 || elem_bytes <= 0) return -1;
  // smallest multiple of (16 / gcd(16, elem_bytes)) elements not below mn
  int g = 16, e = elem_bytes;
  while (e) { int t = g % e; g = e; e = t; }
  const int unit = 16 / g;
  return (mn + unit - 1) / unit * unit;
}

int dg_get_mk_alignment_for_contiguous_layout(void) { return dgk::BLOCK_M; }

const char* dg_last_error_string(void) { return t_err.c_str(); }

dg_status dg_get_device_status(void* stream) {
  DeviceState* st = nullptr;
  int dev = 0;
  dg_status s = device_state(&st, &dev);
  if (s != DG_OK) return s;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  take_status_kernel<<<1, 1, 0, cs>>>();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "status read launch");
  unsigned int v = 0;
  if ((e = cudaMemcpyFromSymbolAsync(&v, g_dg_status_taken, sizeof(v), 0,
                                     cudaMemcpyDeviceToHost, cs)) != cudaSuccess)
    return cuda_fail(e, "read status");
  if ((e = cudaStreamSynchronize(cs)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  switch (v) {
    case dgk::ST_OK: return ok();
    case dgk::ST_TIMEOUT: return fail(DG_ERR_TIMEOUT, "a kernel wait timed out");
    case dgk::ST_MASK_RANGE: return fail(DG_ERR_MASK_RANGE, "masked_m outside [0, max_m]");
    case dgk::ST_EXPERT_RANGE:
      return fail(DG_ERR_EXPERT_RANGE, "m_indices out of range or a block mixes experts");
    case dgk::ST_KS_RANGE:
      return fail(DG_ERR_KS_RANGE, "ks: a negative or partial K group, or past K_total");
    case dgk::ST_DEBUG_BOUNDS:
      return fail(DG_ERR_DEBUG_BOUNDS, "checked build: an access outside a tensor was skipped");
    case dgk::ST_DEBUG_PHASE:
      return fail(DG_ERR_DEBUG_PHASE, "checked build: a ring slot held another fill");
    default: return fail(DG_ERR_CUDA, "unknown device status %u", v);
  }
}

namespace {
dg_status plan_config(int kind, int m, int n, int k, int num_groups, int num_sms, bool sfp,
                      dg_config* out) {
  read_env_once();
  if (!out || kind < 0 || kind > 3 || m < 1 || n < 16 || n % 16 || k < 128 || k % 128 ||
      k > 128 * dgk::MAX_KB || num_sms < 1 || (kind != dgk::kDense && num_groups < 1))
    return fail(DG_ERR_INVALID_ARG, "dg_plan_config: bad arguments");
  const int G = kind == dgk::kDense ? 1 : num_groups;
  // With a GB300 as the current device, clusters fit as the device reports
  // (the configuration a launch takes); otherwise num_sms / S clusters of S.
  DeviceState* st = nullptr;
  {
    int cnt = 0, dev = 0, major = 0, minor = 0;
    if (cudaGetDeviceCount(&cnt) == cudaSuccess && cnt > 0 && cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
        major == 10 && minor == 3) {
      int d = -1;
      if (device_state(&st, &d) != DG_OK || num_sms > st->sms) st = nullptr;
    }
    cudaGetLastError();
  }
  auto cap = [&](int i, const Instance& in, int S, int smem) {
    if (S <= 1) return num_sms;
    return st ? clusters_resident(*st, kind, i, in, S, smem, num_sms) : num_sms / S;
  };
  const int layout = kind == dgk::kKGrouped ? dgk::kTN : dgk::kNT;
  const Plan pl = choose(kind, m, n, k, G, num_sms, cap, g_force_bn.load(), g_force_split.load(),
                         layout, sfp);
  if (pl.inst < 0) return fail(DG_ERR_UNSUPPORTED_SHAPE, "no configuration");
  const Instance& in = table_for(table_id(kind, layout, sfp)).p[pl.inst];
  out->block_m = in.pair ? 2 * dgk::BLOCK_M : dgk::BLOCK_M;
  out->pair = in.pair;
  out->block_n = in.block_n;
  out->split_k = pl.split;
  out->stages = in.stages;
  out->num_tiles = (int)pl.tiles;
  out->grid = std::max(1, pl.clusters) * (pl.pair ? 2 : pl.split);
  out->smem_bytes = pl.smem;
  out->block_scaled = in.bs ? 1 : 0;
  return ok();
}
}  // namespace

dg_status dg_plan_config(int kind, int m, int n, int k, int num_groups, int num_sms,
                         dg_config* out) {
  return plan_config(kind, m, n, k, num_groups, num_sms, false, out);
}

dg_status dg_plan_config_ue8m0(int kind, int m, int n, int k, int num_groups, int num_sms,
                               dg_config* out) {
  return plan_config(kind, m, n, k, num_groups, num_sms, true, out);
}

long long dg_num_output_tiles(int m, int n, int block_m, int block_n) {
  if (block_m <= 0 || block_n <= 0 || m < 0 || n < 0) return -1;
  return cdiv(m, block_m) * cdiv(n, block_n);
}

dg_status dg_set_wait_timeout_ns(unsigned long long ns) {
  g_timeout_ns.store(ns ? ns : 2000000000ull);
  return ok();
}

dg_status dg_debug_set_skip_producer(int on) {
  g_skip_producer.store(on ? 1 : 0);
  return ok();
}

dg_status dg_debug_force_pair(int mode) {
  if (mode < -1 || mode > 1) return fail(DG_ERR_INVALID_ARG, "pair mode %d", mode);
  g_force_pair.store(mode);
  return ok();
}

dg_status dg_debug_force_block_scaled(int mode) {
  if (mode < -1 || mode > 1) return fail(DG_ERR_INVALID_ARG, "block-scaled mode %d", mode);
  read_env_once();
  g_force_bs.store(mode);
  return ok();
}

dg_status dg_debug_force_config(int block_n, int split_k) {
  read_env_once();
  if (block_n < 0 || split_k < 0 || split_k > kMaxCluster)
    return fail(DG_ERR_INVALID_ARG, "block_n=%d split_k=%d", block_n, split_k);
  g_force_bn.store(block_n);
  g_force_split.store(split_k);
  return ok();
}

}  // extern "C"
