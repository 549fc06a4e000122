// i8_api.cu -- the C ABI of libi8 (declared in include/i8.h): argument
// validation, the shape -> kernel-configuration table, TMA descriptors and
// the launches.  The whole library is this one translation unit.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdint>
#include <cstdlib>
#include <atomic>
#include <chrono>
#include <cstring>
#include <mutex>
#include <random>

#include "../../include/i8.h"
#include "gemm.cuh"
#include "gemm_direct.cuh"
#include "gemm_pair.cuh"
#include "producer.cuh"
#include "skinny.cuh"
#include "ptx.cuh"
#include "quant.cuh"

namespace i8 {

// ----------------------------------------------------------------- widen
// int8 codes -> fp16 codes (exact); 16 codes per thread per step.
__global__ void __launch_bounds__(256) widen_codes_kernel(const int8_t* __restrict__ src,
                                                          uint16_t* __restrict__ dst,
                                                          int64_t n16) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + i * 16);
    uint4 o0, o1;
    s8x4_to_f16x4(v.x, o0.x, o0.y);
    s8x4_to_f16x4(v.y, o0.z, o0.w);
    s8x4_to_f16x4(v.z, o1.x, o1.y);
    s8x4_to_f16x4(v.w, o1.z, o1.w);
    reinterpret_cast<uint4*>(dst + i * 16)[0] = o0;
    reinterpret_cast<uint4*>(dst + i * 16)[1] = o1;
  }
}

// Failure-detection self-test: one thread waits on an mbarrier that nothing
// ever arrives at, through the same bounded wait the GEMM pipeline uses.  The
// wait gives up after limit_ns, records I8_ERR_DEVICE_TIMEOUT in the status
// word and the kernel returns normally (no trap, no fault, no hang).
__global__ void selftest_timeout_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  abort_flag = 0;
  fence_mbarrier_init();
  mbar_wait(b, 0u, &abort_flag, limit_ns);
}

namespace {

constexpr int kMaxDevices = 64;

// Process-wide tuning knobs (i8_set_option).
struct Options {
  int chunk_k = 1024;      // K per exact fp32 chunk (multiple of 64, <= 1024)
  int force_splits = 0;    // 0 = table
  int max_ctas = 0;        // 0 = all SMs
  int force_bn = 0;        // 0 = table, else 128 or 256
  int quant_vpl = 6;       // max 16-byte vectors per lane in the quantizer
  int cta_pair = 0;        // 0 = table, 1 = never, 2 = whenever the shape allows
  int skinny_max_m = 16;   // token counts up to this use the weight-streaming kernel (0 = off)
  int pdl = 1;             // launch with programmatic stream serialization
  int quant_rows = 0;      // quantizer rows per CTA (0 = by shape)
  int stream_k = 1;        // CTA-pair stream-K: 0 never, 1 by the table, 2 whenever pairs idle
  int nvtx = 0;            // NVTX range around every ABI call
  int pair_stage_k = 0;    // K per fp16 stage of the int8-code pair kernel: 0 (table) / 64 / 128
  int raster = 0;          // tile order: 0 table, 1 M blocks fastest, 2 N blocks fastest
};
Options g_opt;

// NVTX range for the lifetime of one ABI call (when I8_OPT_NVTX is on).
struct NvtxScope {
  bool on;
  explicit NvtxScope(const char* name) : on(g_opt.nvtx != 0) {
    if (on) nvtxRangePushA(name);
  }
  ~NvtxScope() {
    if (on) nvtxRangePop();
  }
};
#define I8_NVTX() NvtxScope i8_nvtx_scope_(__func__)

struct DeviceInfo {
  bool init = false;
  int sms = 0;
  int pair_clusters[4] = {};  // co-resident clusters per pair-kernel config
  int cc_major = 0, cc_minor = 0;
  bool smem_set[12] = {};
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

i8_status cuda_status(cudaError_t e) { return e == cudaSuccess ? I8_OK : I8_ERR_CUDA; }

i8_status device_info(DeviceInfo** out, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return I8_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return I8_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
            cudaSuccess)
      return I8_ERR_CUDA;
    d.init = true;
  }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return I8_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *out = &d;
  if (dev_out) *dev_out = dev;
  return I8_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with programmatic stream serialization (unless switched off): the
// kernel may be scheduled while the previous kernel of the stream drains.
// Every kernel launched this way calls pdl_wait() before it touches global
// memory, so the stream order of memory effects is unchanged.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g_opt.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// ----------------------------------------------------------------- quant
template <int V>
cudaError_t launch_quant_v(const uint16_t* x, int64_t rows, int K, int64_t ldx, int8_t* q,
                           int64_t ldq, float* s, int G, int R, int fmt, cudaStream_t st) {
  const int64_t grid = (rows + R - 1) / R;
  if (fmt == kQuantE4M3)
    return launch_pdl(quant_rows_kernel<V, kQuantE4M3>, dim3(static_cast<unsigned>(grid)),
                      dim3(32 * G * R), 0, st, x, rows, K, ldx, q, ldq, s, G);
  if (fmt == kQuantF16)
    return launch_pdl(quant_rows_kernel<V, kQuantF16>, dim3(static_cast<unsigned>(grid)),
                      dim3(32 * G * R), 0, st, x, rows, K, ldx, q, ldq, s, G);
  return launch_pdl(quant_rows_kernel<V>, dim3(static_cast<unsigned>(grid)), dim3(32 * G * R), 0,
                    st, x, rows, K, ldx, q, ldq, s, G);
}

// fmt: kQuantInt8 (int8 codes), kQuantE4M3 (E4M3 bit patterns) or kQuantF16
// (the int8 codes as fp16 values; ldq then counts fp16 elements).
i8_status quant_rows(const void* x, int64_t rows, int64_t K, int64_t ldx, int8_t* q, int64_t ldq,
                     float* s, cudaStream_t st, int fmt = kQuantInt8) {
  if (rows < 0 || K <= 0 || ldx < K || ldq < K) return I8_ERR_INVALID_ARG;
  if (rows > 0 && (!x || !q || !s)) return I8_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > 131072 || rows > INT32_MAX) return I8_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(q) || !aligned4(s) || ldx % 8 != 0 ||
      ldq % (fmt == kQuantF16 ? 8 : 16) != 0)
    return I8_ERR_ALIGNMENT;
  if (rows == 0) return I8_OK;
  DeviceInfo* d;
  if (i8_status e = device_info(&d, nullptr)) return e;
  // Vectors of 8 elements per row; G warps per row, V vectors per lane.
  const int vecs = static_cast<int>(K / 8);
  int G = 1;
  while (G < 8 && (vecs + 32 * G - 1) / (32 * G) > g_opt.quant_vpl) G *= 2;
  const int need = (vecs + 32 * G - 1) / (32 * G);
  // R rows per CTA (G * R <= 8 warps).  One row per CTA by default: the
  // smallest CTAs balance best across the SMs (measured 7-11 % faster than
  // 8 / G rows per CTA at the DiT shapes, never slower).
  const int R = g_opt.quant_rows > 0 ? std::min(g_opt.quant_rows, 8 / G) : 1;
  const auto* xb = static_cast<const uint16_t*>(x);
  const int Ki = static_cast<int>(K);
  cudaError_t e;
  if (need > 16) {
    // longer than 8 warps x 32 lanes x 16 vectors: the two-pass kernel
    if (fmt == kQuantE4M3)
      e = launch_pdl(quant_rows_long_kernel<kQuantE4M3>, dim3(static_cast<unsigned>(rows)),
                     dim3(256), 0, st, xb, rows, Ki, ldx, q, ldq, s);
    else if (fmt == kQuantF16)
      e = launch_pdl(quant_rows_long_kernel<kQuantF16>, dim3(static_cast<unsigned>(rows)),
                     dim3(256), 0, st, xb, rows, Ki, ldx, q, ldq, s);
    else
      e = launch_pdl(quant_rows_long_kernel<kQuantInt8>, dim3(static_cast<unsigned>(rows)),
                     dim3(256), 0, st, xb, rows, Ki, ldx, q, ldq, s);
    return cuda_status(e);
  }
  if (need <= 1) e = launch_quant_v<1>(xb, rows, Ki, ldx, q, ldq, s, G, R, fmt, st);
  else if (need <= 2) e = launch_quant_v<2>(xb, rows, Ki, ldx, q, ldq, s, G, R, fmt, st);
  else if (need <= 3) e = launch_quant_v<3>(xb, rows, Ki, ldx, q, ldq, s, G, R, fmt, st);
  else if (need <= 4) e = launch_quant_v<4>(xb, rows, Ki, ldx, q, ldq, s, G, R, fmt, st);
  else if (need <= 6) e = launch_quant_v<6>(xb, rows, Ki, ldx, q, ldq, s, G, R, fmt, st);
  else if (need <= 8) e = launch_quant_v<8>(xb, rows, Ki, ldx, q, ldq, s, G, R, fmt, st);
  else if (need <= 12) e = launch_quant_v<12>(xb, rows, Ki, ldx, q, ldq, s, G, R, fmt, st);
  else e = launch_quant_v<16>(xb, rows, Ki, ldx, q, ldq, s, G, R, fmt, st);  // need <= 16
  return cuda_status(e);
}

// ----------------------------------------------------------------- producer + quant
template <int V, int FMT>
cudaError_t launch_producer_v(int op, const uint16_t* x, int64_t rows, int K, int64_t ldx,
                              float eps, int8_t* q, int64_t ldq, float* s, uint16_t* y,
                              int64_t ldy, int G, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(rows)), block(32 * G);
  if (op == kOpLayerNorm)
    return launch_pdl(producer_quant_kernel<V, FMT, kOpLayerNorm>, grid, block, 0, st, x, rows, K,
                      ldx, eps, q, ldq, s, y, ldy, G);
  return launch_pdl(producer_quant_kernel<V, FMT, kOpGelu>, grid, block, 0, st, x, rows, K, ldx,
                    eps, q, ldq, s, y, ldy, G);
}

template <int FMT>
cudaError_t launch_producer(int op, const uint16_t* x, int64_t rows, int K, int64_t ldx, float eps,
                            int8_t* q, int64_t ldq, float* s, uint16_t* y, int64_t ldy, int need,
                            int G, cudaStream_t st) {
  if (need <= 1) return launch_producer_v<1, FMT>(op, x, rows, K, ldx, eps, q, ldq, s, y, ldy, G, st);
  if (need <= 2) return launch_producer_v<2, FMT>(op, x, rows, K, ldx, eps, q, ldq, s, y, ldy, G, st);
  if (need <= 3) return launch_producer_v<3, FMT>(op, x, rows, K, ldx, eps, q, ldq, s, y, ldy, G, st);
  if (need <= 4) return launch_producer_v<4, FMT>(op, x, rows, K, ldx, eps, q, ldq, s, y, ldy, G, st);
  if (need <= 6) return launch_producer_v<6, FMT>(op, x, rows, K, ldx, eps, q, ldq, s, y, ldy, G, st);
  if (need <= 8) return launch_producer_v<8, FMT>(op, x, rows, K, ldx, eps, q, ldq, s, y, ldy, G, st);
  if (need <= 12) return launch_producer_v<12, FMT>(op, x, rows, K, ldx, eps, q, ldq, s, y, ldy, G, st);
  return launch_producer_v<16, FMT>(op, x, rows, K, ldx, eps, q, ldq, s, y, ldy, G, st);
}

// The GELU table is built once per device, by the first GELU call, on that
// call's stream, which is then synchronized (so the first call must not be
// made during stream capture).
bool g_gelu_table_ready[kMaxDevices] = {};

i8_status ensure_gelu_table(cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return I8_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_gelu_table_ready[dev]) return I8_OK;
  gelu_table_kernel<<<65536 / 256, 256, 0, st>>>();
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return I8_ERR_CUDA;
  g_gelu_table_ready[dev] = true;
  return I8_OK;
}

template <int V, int FMT>
cudaError_t launch_gelu_table_v(const uint16_t* x, int64_t rows, int K, int64_t ldx, int8_t* q,
                                int64_t ldq, float* s, uint16_t* y, int64_t ldy, int G, int sms,
                                cudaStream_t st) {
  auto kern = gelu_table_quant_kernel<V, FMT>;
  constexpr int kSmem = 65536 * 2;   // the table
  static bool smem_set[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!smem_set[dev]) {
      const cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      if (e != cudaSuccess) return e;
      smem_set[dev] = true;
    }
  }
  const int R = 16 / G;
  const int64_t groups = (rows + R - 1) / R;
  const int grid = static_cast<int>(std::min<int64_t>(groups, sms));
  return launch_pdl(kern, dim3(grid), dim3(512), kSmem, st, x, rows, K, ldx, q, ldq, s, y, ldy, G);
}

template <int FMT>
cudaError_t launch_gelu_table(const uint16_t* x, int64_t rows, int K, int64_t ldx, int8_t* q,
                              int64_t ldq, float* s, uint16_t* y, int64_t ldy, int need, int G,
                              int sms, cudaStream_t st) {
  if (need <= 1) return launch_gelu_table_v<1, FMT>(x, rows, K, ldx, q, ldq, s, y, ldy, G, sms, st);
  if (need <= 2) return launch_gelu_table_v<2, FMT>(x, rows, K, ldx, q, ldq, s, y, ldy, G, sms, st);
  if (need <= 3) return launch_gelu_table_v<3, FMT>(x, rows, K, ldx, q, ldq, s, y, ldy, G, sms, st);
  if (need <= 4) return launch_gelu_table_v<4, FMT>(x, rows, K, ldx, q, ldq, s, y, ldy, G, sms, st);
  if (need <= 6) return launch_gelu_table_v<6, FMT>(x, rows, K, ldx, q, ldq, s, y, ldy, G, sms, st);
  if (need <= 8) return launch_gelu_table_v<8, FMT>(x, rows, K, ldx, q, ldq, s, y, ldy, G, sms, st);
  if (need <= 12) return launch_gelu_table_v<12, FMT>(x, rows, K, ldx, q, ldq, s, y, ldy, G, sms, st);
  return launch_gelu_table_v<16, FMT>(x, rows, K, ldx, q, ldq, s, y, ldy, G, sms, st);
}

// LayerNorm / GELU of each row, then the per-row quantizer of the bf16
// result; y (optional) receives that bf16 result.  Rows must fit the
// register-resident layout: K <= 32768.
i8_status producer_quant(int op, const void* x, int64_t rows, int64_t K, int64_t ldx, float eps,
                         int fmt, void* q, int64_t ldq, float* s, void* y, int64_t ldy,
                         cudaStream_t st) {
  if (rows < 0 || K <= 0 || ldx < K || ldq < K || (y && ldy < K)) return I8_ERR_INVALID_ARG;
  if (fmt != kQuantInt8 && fmt != kQuantE4M3 && fmt != kQuantF16) return I8_ERR_INVALID_ARG;
  if (op == kOpLayerNorm && !(eps >= 0.0f && eps <= 3.0e38f)) return I8_ERR_INVALID_ARG;
  if (rows > 0 && (!x || !q || !s)) return I8_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > 32768 || rows > INT32_MAX) return I8_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(q) || !aligned4(s) || ldx % 8 != 0 ||
      ldq % (fmt == kQuantF16 ? 8 : 16) != 0 || (y && (!aligned16(y) || ldy % 8 != 0)))
    return I8_ERR_ALIGNMENT;
  if (rows == 0) return I8_OK;
  DeviceInfo* d;
  if (i8_status e = device_info(&d, nullptr)) return e;
  const int vecs = static_cast<int>(K / 8);
  int G = 1;
  while (G < 8 && (vecs + 32 * G - 1) / (32 * G) > g_opt.quant_vpl) G *= 2;
  const int need = (vecs + 32 * G - 1) / (32 * G);
  const auto* xb = static_cast<const uint16_t*>(x);
  auto* qb = static_cast<int8_t*>(q);
  auto* yb = static_cast<uint16_t*>(y);
  const int Ki = static_cast<int>(K);
  if (op == kOpGelu) {
    if (i8_status e = ensure_gelu_table(st)) return e;
    const cudaError_t e =
        fmt == kQuantE4M3
            ? launch_gelu_table<kQuantE4M3>(xb, rows, Ki, ldx, qb, ldq, s, yb, ldy, need, G, d->sms, st)
        : fmt == kQuantF16
            ? launch_gelu_table<kQuantF16>(xb, rows, Ki, ldx, qb, ldq, s, yb, ldy, need, G, d->sms, st)
            : launch_gelu_table<kQuantInt8>(xb, rows, Ki, ldx, qb, ldq, s, yb, ldy, need, G, d->sms, st);
    return cuda_status(e);
  }
  const cudaError_t e =
      fmt == kQuantE4M3
          ? launch_producer<kQuantE4M3>(op, xb, rows, Ki, ldx, eps, qb, ldq, s, yb, ldy, need, G, st)
      : fmt == kQuantF16
          ? launch_producer<kQuantF16>(op, xb, rows, Ki, ldx, eps, qb, ldq, s, yb, ldy, need, G, st)
          : launch_producer<kQuantInt8>(op, xb, rows, Ki, ldx, eps, qb, ldq, s, yb, ldy, need, G, st);
  return cuda_status(e);
}

// Stream-K launch tags: a process-wide counter started at a random 48-bit
// value, so a launch's tag differs from every earlier launch's (whose words
// may still sit in a reused workspace) and, with overwhelming probability,
// from whatever a fresh workspace holds.
unsigned long long next_sk_epoch() {
  static std::atomic<unsigned long long> counter{[] {
    std::random_device rd;
    const unsigned long long t = static_cast<unsigned long long>(
        std::chrono::steady_clock::now().time_since_epoch().count());
    return ((static_cast<unsigned long long>(rd()) << 32) ^ rd() ^ t) & ((1ull << 48) - 1);
  }()};
  unsigned long long e;
  do {
    e = counter.fetch_add(1) & ((1ull << 48) - 1);
  } while (e == 0);
  return e;
}

// ----------------------------------------------------------------- GEMM plan
struct Plan {
  bool skinny = false;     // few tokens: weight-streaming kernel
  bool pair = false;       // CTA-pair kernel (256 x 256 tiles per cluster of 2)
  bool stream_k = false;   // pair kernel with the stream-K schedule
  int sk_waves = 0;        // stream-K: whole waves of tiles before the split ones
  int sk_pairs = 0;        // stream-K: pairs sharing the split tiles' units
  size_t sk_arrive_bytes = 0;  // stream-K: arrival words at the start of ws
  int bn = 128;
  int splits = 1;
  int kb_per_split = 1;
  int total_kb = 1;
  int num_m = 1, num_n = 1;
  int num_tiles = 1;
  int grid = 1;
  int chunk_stages = 8;
  int n_fastest = 0;       // tile order: 1 N blocks fastest, 0 M blocks
  int64_t ws_ld = 0;       // row stride of the split partials (elements)
  size_t ws_bytes = 0;
};

// K-splits for `tiles` output tiles on `slots` concurrent workers: the
// smallest split count that maximises the filled fraction of the last wave,
// with at least 4 K-blocks (512 K) per split; 1 when the tiles already fill
// every worker.
int best_splits(int64_t tiles, int slots, int total_kb) {
  if (tiles >= slots) return 1;
  int best = 1;
  double best_eff = static_cast<double>(tiles) / slots;
  const int max_s = std::max(1, std::min(16, total_kb / 4));
  for (int s = 2; s <= max_s; ++s) {
    const int64_t items = tiles * s;
    const int64_t rounds = (items + slots - 1) / slots;
    const double eff = static_cast<double>(items) / static_cast<double>(rounds * slots);
    if (eff > best_eff + 1e-9) {
      best = s;
      best_eff = eff;
    }
  }
  return best;
}

// Tile order.  The tiles running at the same time share weight columns when
// M blocks run fastest and activation rows when N blocks do; the reused
// operand should be the larger one, which must otherwise be re-read from HBM
// once it outgrows L2 (MLP down-projection, 8704 x 12288 activations: M-fastest
// read 513 MB from DRAM per call for 145 MB of operands).
int tile_order_n_fastest(int64_t M, int64_t N) {
  if (g_opt.raster != 0) return g_opt.raster == 2 ? 1 : 0;
  return M > N ? 1 : 0;
}

// Few tokens: the weight-streaming kernel (any code format), which measured
// 1.4-2.2x faster than the tiled kernels with K splits at every M <= 16 of
// the DiT sweep (e.g. 16 x 3072 x 9216: 10.4 against 20.1 us; 8 x 3072 x
// 18432: 13.2 against 27.6 us).
// What one few-token kernel variant can hold on the device at once: its
// resident CTA slots, and for each cluster size s the clusters of s CTAs
// resident together (0 where unknown: slots / s).  A cluster sits within one
// GPC, so with one CTA per SM fewer fit than slots / s (GB300, 152 SMs, one
// CTA per SM: 46 clusters of 3, 36 of 4, 15 of 8).
struct SkinnyFit {
  int slots = 0;
  int clusters[kSkinnyMaxSplits + 1] = {};
  int cap(int s) const { return clusters[s] > 0 ? clusters[s] : slots / s; }
};

// Few-token split planning: least 256-K stages per K split (512 K), and the
// stages per CTA above which K counts as long.
constexpr int kSkinnySplitMinStages = 2;
constexpr int kSkinnyLongStages = 12;

void plan_skinny(Plan& p, int64_t M, int64_t N, int64_t K, int sms, const SkinnyFit& fit) {
  (void)M;
  // K splits, when the N-blocks leave more than a tenth of the SMs idle.
  // Short K: the fewest that give about 5/8 of the SMs a CTA; every CTA
  // carries a fixed cost (start, epilogue, its share of the cluster's
  // reduction) that more, shorter CTAs would not repay.  Long K (more than
  // kSkinnyLongStages stages per CTA that way): the fewest that give every
  // SM a CTA, since one CTA alone streams no faster than about 25-50 GB/s.
  // Then at most kSkinnyMaxSplits, at least kSkinnySplitMinStages whole
  // 256-K stages per split, and lowered until all CTAs are resident at once
  // (within the CTA slots, and the N-blocks' clusters within the clusters
  // that fit; a second wave would stream its weights only after the first
  // finished).  One N-block's splits form a cluster.  No workspace: the
  // splits add their partials over distributed shared memory.
  // Measured (GB300, graph replay, weights rotating past L2; M x K x N,
  // int8 codes, us with 1 / 2 / 3 / 4 / 6 splits):
  //   * 16 x 3072 x 3072: 8.5 / 5.9 / 6.7 / 6.9 / 11.6 (48 N-blocks);
  //   * 1 x 3072 x 768: 6.1 / 4.1 / 3.6 / 3.2 / 2.9 (12 N-blocks);
  //   * 1 x 2048 x 6144: 4.8 / 5.2 / 5.6 / 7.1 (96 N-blocks);
  //   * 1 x 12288 x 3072: 23.2 / 13.1 / 13.2 / 11.1 / 14.3 (long K; with 6
  //     the 48 clusters no longer fit at once);
  //   * 16 x 12288 x 3072, fp16-held codes (one CTA per SM): 29.6 / 18.8 /
  //     27.2 / 22.8 with 1 / 2 / 3 / 4 (46 clusters of 3 fit, not 48).
  p.skinny = true;
  p.num_n = static_cast<int>((N + kSkinnyRows - 1) / kSkinnyRows);
  p.num_m = 1;
  const int stages = static_cast<int>((K + kSkinnyK - 1) / kSkinnyK);
  int splits = 1;
  if (g_opt.force_splits > 0) {
    splits = g_opt.force_splits;
  } else if (10LL * p.num_n < 9LL * sms) {
    const int short_ctas = std::max(1, 5 * sms / 8);
    splits = (short_ctas + p.num_n - 1) / p.num_n;
    if ((stages + splits - 1) / splits > kSkinnyLongStages) splits = (sms + p.num_n - 1) / p.num_n;
    splits = std::min(splits, std::max(1, stages / kSkinnySplitMinStages));
    splits = std::min(splits, kSkinnyMaxSplits);
    while (splits > 1 &&
           (static_cast<int64_t>(p.num_n) * splits > fit.slots || p.num_n > fit.cap(splits)))
      --splits;
  }
  splits = std::max(1, std::min(std::min(splits, stages), kSkinnyMaxSplits));
  p.kb_per_split = (stages + splits - 1) / splits;          // stages per split
  p.splits = (stages + p.kb_per_split - 1) / p.kb_per_split;
  p.total_kb = stages;
  p.grid = p.num_n * p.splits;
}

// Shape -> configuration (replaces per-shape autotuning).
//   * few tokens (M <= 16 by default): the weight-streaming kernel;
//   * CTA pairs (one 256 x 256 tile per cluster of two SMs, each SM staging
//     and widening half of B) for int8 weights whenever M, N >= 256; with
//     pre-widened weights the single-CTA kernel measured slightly faster;
//   * otherwise one CTA per 128 x 256 tile (128 x 128 when the wider tiles
//     would leave SMs idle);
//   * stream-K on CTA pairs by the rule below, else split-K (exact int32
//     partials + a reduction) when the tiles cannot fill every worker;
//   * the tile order from tile_order_n_fastest (M blocks fastest under
//     stream-K unless the raster option sets it), applied by the caller.
Plan make_plan(int64_t M, int64_t N, int64_t K, int sms, int pair_clusters = 0,
               bool b16 = false, size_t ws_cap = SIZE_MAX, SkinnyFit fit = SkinnyFit()) {
  Plan p;
  p.n_fastest = tile_order_n_fastest(M, N);
  if (pair_clusters <= 0) pair_clusters = sms / 2;
  if (fit.slots <= 0) fit.slots = 2 * sms;
  p.total_kb = static_cast<int>((K + 127) / 128);
  if (M <= g_opt.skinny_max_m) {
    plan_skinny(p, M, N, K, sms, fit);
    return p;
  }
  const bool pair_ok = M >= 256 && N >= 256;
  p.pair = g_opt.cta_pair == 2 ? pair_ok : (g_opt.cta_pair == 0 && !b16 && pair_ok);
  int64_t tiles;
  int slots;
  if (p.pair) {
    p.bn = 256;
    p.num_m = static_cast<int>((M + 255) / 256);
    p.num_n = static_cast<int>((N + 255) / 256);
    tiles = static_cast<int64_t>(p.num_m) * p.num_n;
    slots = pair_clusters;
    if (g_opt.max_ctas > 0) slots = std::max(1, std::min(slots, g_opt.max_ctas / 2));
    // Stream-K: every pair gets an equal share of the (tile, K-block)
    // units, at least 4 K-blocks each.  Workspace: one arrival word per
    // (tile, CTA) and one 256 x 256 int32 partial slot per pair.  A pair's
    // schedule then holds one item more than its share of whole tiles, and
    // the tile it finishes last waits for one or two partials to load: about
    // 6-9 us per launch against whole tiles at K = 3072.  The table takes it
    // where whole tiles leave more than that idle: at least half a wave of
    // tiles and a whole-tile wave efficiency below 0.93.  Plans that split
    // every tile take the M-blocks-fastest tile order, which measured as
    // fast or faster there at every shape with M > N; plans with whole waves
    // first take the table's order (N-blocks fastest when M > N: MLP
    // down-projection 431.2 against 442.4 us).
    // Measured (GEMM, GB300, 30 DiT sweep shapes): every shape the rule
    // takes gains 1-12 % (e.g. 1024 x 3072 x 3072 32.8 -> 30.3 us,
    // 4096 x 3072 x 12288 230 -> 212 us, 1024 x 3072 x 12288 103 -> 66 us)
    // but one, 16384 x 3072 x 12288 (820.0 -> 821.6 us); at a wave
    // efficiency of 0.95 and above stream-K loses up to 9 %, and with 12 or
    // 36 tiles split-K is faster.
    const int64_t units = tiles * p.total_kb;
    const int64_t waves = (tiles + slots - 1) / slots;
    const double wave_eff = static_cast<double>(tiles) / static_cast<double>(waves * slots);
    const bool sk_table = 2 * tiles >= slots && wave_eff < 0.93;
    if ((g_opt.stream_k == 2 || (g_opt.stream_k == 1 && sk_table)) && g_opt.force_splits == 0 &&
        tiles % slots != 0 &&
        units * slots < (int64_t(1) << 31)) {   // the kernel's unit arithmetic is 32-bit
      // Long K (>= 64 K-blocks): whole waves of tiles first (tile = pair +
      // wave * pairs, neighbours in flight together), then only the
      // remaining tiles' units split evenly.  Shorter K: every tile's units
      // split evenly.  At least 4 K-blocks per pair either way.
      // Measured (GEMM, GB300, both schedules forced, one process): whole
      // waves first gained 2-14 % at K = 12288 (MLP down-projection 445.2 ->
      // 431.2 us, 16384 x 3072 x 12288 857 -> 804 us, with the table's tile
      // order) and lost 1-7 % at K = 3072 (QKV 106.7 -> 109.9 us).
      const int64_t dp_waves = p.total_kb >= 64 ? tiles / slots : 0;
      const int pairs = dp_waves > 0 ? slots
                                     : static_cast<int>(std::min<int64_t>(slots, std::max<int64_t>(1, units / 4)));
      const int64_t sk_units = (tiles - dp_waves * pairs) * p.total_kb;
      const int sk_pairs = static_cast<int>(std::min<int64_t>(pairs, std::max<int64_t>(1, sk_units / 4)));
      const size_t arrive = (static_cast<size_t>(tiles) * 16 + 1023) / 1024 * 1024;
      const size_t part = static_cast<size_t>(sk_pairs) * 256 * 256 * sizeof(int32_t);
      if (arrive + part <= ws_cap) {
        p.stream_k = true;
        p.sk_waves = static_cast<int>(dp_waves);
        p.sk_pairs = sk_pairs;
        p.n_fastest = g_opt.raster != 0 ? (g_opt.raster == 2 ? 1 : 0)
                                        : (dp_waves > 0 ? tile_order_n_fastest(M, N) : 0);
        p.num_tiles = static_cast<int>(tiles);
        p.kb_per_split = p.total_kb;
        p.grid = 2 * pairs;
        p.chunk_stages = g_opt.chunk_k / 64;
        p.sk_arrive_bytes = arrive;
        p.ws_bytes = arrive + part;
        return p;
      }
    }
  } else {
    p.bn = (N >= 256 && ((M + 127) / 128) * ((N + 255) / 256) >= sms) ? 256 : 128;
    if (g_opt.force_bn == 128 || g_opt.force_bn == 256) p.bn = g_opt.force_bn;
    p.num_m = static_cast<int>((M + 127) / 128);
    p.num_n = static_cast<int>((N + p.bn - 1) / p.bn);
    tiles = static_cast<int64_t>(p.num_m) * p.num_n;
    slots = g_opt.max_ctas > 0 ? std::min(g_opt.max_ctas, sms) : sms;
  }
  int splits = g_opt.force_splits > 0 ? g_opt.force_splits : best_splits(tiles, slots, p.total_kb);
  splits = std::max(1, std::min(splits, p.total_kb));
  p.kb_per_split = (p.total_kb + splits - 1) / splits;
  p.splits = (p.total_kb + p.kb_per_split - 1) / p.kb_per_split;
  // A capped workspace (the no-alloc entry's fixed array): fewer splits until
  // the int32 partial planes fit, down to one split, which needs none.
  if (g_opt.force_splits == 0) {
    const size_t plane = static_cast<size_t>(M) * static_cast<size_t>((N + 3) / 4 * 4) * 4;
    while (p.splits > 1 && static_cast<size_t>(p.splits) * plane > ws_cap) {
      splits = p.splits - 1;
      p.kb_per_split = (p.total_kb + splits - 1) / splits;
      p.splits = (p.total_kb + p.kb_per_split - 1) / p.kb_per_split;
    }
  }
  p.num_tiles = static_cast<int>(tiles * p.splits);
  p.grid = std::max(1, static_cast<int>(std::min<int64_t>(p.num_tiles, slots)));
  if (p.pair) p.grid *= 2;
  p.chunk_stages = g_opt.chunk_k / 64;
  if (p.splits > 1) {
    p.ws_ld = (N + 3) / 4 * 4;
    p.ws_bytes = static_cast<size_t>(p.splits) * static_cast<size_t>(M) *
                 static_cast<size_t>(p.ws_ld) * sizeof(int32_t);
  }
  return p;
}

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output map for the epilogue's bulk tensor stores: {N, M, planes} with the
// split-K partial index as the third coordinate; 128-byte-wide boxes of 32 rows.
bool encode_out(CUtensorMap* map, bool bf16, const void* base, uint64_t N, uint64_t M,
                uint64_t ld_elems, uint64_t planes) {
  const uint64_t esz = bf16 ? 2 : 4;
  const cuuint64_t dims[3] = {N, M, planes};
  const cuuint64_t strides[2] = {ld_elems * esz, ld_elems * esz * M};
  const cuuint32_t box[3] = {bf16 ? 64u : 32u, 32u, 1u};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_INT32, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class Cfg>
i8_status launch_gemm_cfg(DeviceInfo* d, int slot, const CUtensorMap& ma, const CUtensorMap& mb,
                          const CUtensorMap& my, const GemmParams& gp, int grid, cudaStream_t st) {
  auto kern = gemm_w8a8_kernel<Cfg>;
  if (!d->smem_set[slot]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM_BYTES) != cudaSuccess)
      return I8_ERR_CUDA;
    d->smem_set[slot] = true;
  }
  return cuda_status(launch_pdl(kern, dim3(grid), dim3(Cfg::THREADS), Cfg::SMEM_BYTES, st, ma, mb,
                                my, gp));
}

// <BN, int8 stages, fp16 stages, widen A on chip, widen B on chip>
template <class Cfg>
int pair_cluster_capacity(DeviceInfo* d, int slot) {
  if (d->pair_clusters[slot] > 0) return d->pair_clusters[slot];
  auto kern = gemm_w8a8_pair_kernel<Cfg>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (d->sms / 2), 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  if (n <= 0) n = d->sms / 2;
  d->pair_clusters[slot] = n;
  return n;
}

template <class Cfg>
i8_status launch_pair_cfg(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& my,
                          const CUtensorMap& mp, const GemmParams& gp, int grid, cudaStream_t st) {
  auto kern = gemm_w8a8_pair_kernel<Cfg>;
  return cuda_status(launch_pdl(kern, dim3(grid), dim3(Cfg::THREADS), Cfg::SMEM_BYTES, st, ma, mb,
                                my, mp, gp));
}

// The skinny kernel for the code formats KIND (SkinnyKind) and MT groups of
// 8 tokens: its shared-memory size is set once per device (slots 4..11 of
// smem_set).
template <int KIND, int MT>
bool skinny_prepare(DeviceInfo* d) {
  const int slot = 4 + 2 * KIND + (MT - 1);
  if (!d->smem_set[slot]) {
    if (cudaFuncSetAttribute(gemm_skinny_kernel<KIND, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SkinnyCfg<KIND, MT>::SMEM_BYTES) != cudaSuccess)
      return false;
    d->smem_set[slot] = true;
  }
  return true;
}

// CTA slots and cluster capacities of one skinny kernel variant on this
// device (its split choice keeps the grid within one wave), queried once.
template <int KIND, int MT>
SkinnyFit skinny_fit_of(DeviceInfo* d) {
  static SkinnyFit cached[kMaxDevices];
  static std::atomic<int> ready[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    SkinnyFit f;
    f.slots = d->sms;
    return f;
  }
  if (ready[dev].load(std::memory_order_acquire)) return cached[dev];
  std::lock_guard<std::mutex> lock(mu);
  if (!ready[dev].load(std::memory_order_relaxed)) {
    SkinnyFit f;
    int n = 0;
    if (skinny_prepare<KIND, MT>(d)) {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemm_skinny_kernel<KIND, MT>,
                                                        SkinnyCfg<KIND, MT>::THREADS,
                                                        SkinnyCfg<KIND, MT>::SMEM_BYTES) != cudaSuccess)
        n = 0;
      for (int s = 1; s <= kSkinnyMaxSplits; ++s) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(s, 1, 1);
        cfg.blockDim = dim3(SkinnyCfg<KIND, MT>::THREADS, 1, 1);
        cfg.dynamicSmemBytes = SkinnyCfg<KIND, MT>::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = s;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, gemm_skinny_kernel<KIND, MT>, &cfg) != cudaSuccess) c = 0;
        f.clusters[s] = c;
      }
    }
    cudaGetLastError();
    f.slots = (n > 0 ? n : 1) * d->sms;
    cached[dev] = f;
    ready[dev].store(1, std::memory_order_release);
  }
  return cached[dev];
}
template <int KIND>
SkinnyFit skinny_fit_k(DeviceInfo* d, int64_t M) {
  return M > 8 ? skinny_fit_of<KIND, 2>(d) : skinny_fit_of<KIND, 1>(d);
}
SkinnyFit skinny_fit(DeviceInfo* d, bool b16, int64_t M) {
  return b16 ? skinny_fit_k<kSkW16>(d, M) : skinny_fit_k<kSkI8>(d, M);
}

template <int KIND, int MT>
cudaError_t launch_skinny(DeviceInfo* d, const CUtensorMap& mw, const CUtensorMap& ma,
                          const SkinnyParams& sp, int grid, cudaStream_t st) {
  using Cfg = SkinnyCfg<KIND, MT>;
  if (!skinny_prepare<KIND, MT>(d)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeClusterDimension;   // one N-block's K splits
  attr[n].val.clusterDim.x = static_cast<unsigned>(sp.splits);
  attr[n].val.clusterDim.y = 1;
  attr[n].val.clusterDim.z = 1;
  ++n;
  if (g_opt.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(n);
  return cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<KIND, MT>, mw, ma, sp);
}

// The few-token route for any code format: tensor maps of the weights and
// the token codes, then one launch (the plan from plan_skinny).  out_mode
// kOutInt32 writes the raw accumulator: int32, or fp32 for E4M3.
template <int KIND>
i8_status skinny_route(DeviceInfo* d, const Plan& pl, const void* aq, const void* wb, int64_t M,
                       int64_t N, int64_t K, int out_mode, void* out, int64_t ldo,
                       const float* s_a, const float* s_w, const void* bias, cudaStream_t st) {
  constexpr bool W_F16 = SkinnyCfg<KIND, 1>::W_F16;
  constexpr bool A_F16 = SkinnyCfg<KIND, 1>::A_F16;
  CUtensorMap mw, ma;
  if (!encode_2d(&mw, W_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, wb, K, N,
                 W_F16 ? 2 * K : K, W_F16 ? 64 : 128, kSkinnyRows))
    return I8_ERR_CUDA;
  const int mt = M > 8 ? 2 : 1;   // token groups of 8 (M <= 16)
  if (!encode_2d(&ma, A_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, aq, K, M,
                 A_F16 ? 2 * K : K, A_F16 ? 64 : 128, 8 * mt))
    return I8_ERR_CUDA;
  SkinnyParams sp{};
  sp.M = static_cast<int>(M);
  sp.N = static_cast<int>(N);
  sp.K = static_cast<int>(K);
  sp.num_ks = pl.total_kb;
  sp.ks_per_cta = pl.kb_per_split;
  sp.splits = pl.splits;
  sp.out_mode = out_mode;
  sp.s_a = s_a;
  sp.s_w = s_w;
  sp.bias = static_cast<const uint16_t*>(bias);
  sp.out = out;
  sp.ldo = ldo;
  const cudaError_t le = mt == 2 ? launch_skinny<KIND, 2>(d, mw, ma, sp, pl.grid, st)
                                 : launch_skinny<KIND, 1>(d, mw, ma, sp, pl.grid, st);
  if (le != cudaSuccess) return cuda_status(le);
  return cuda_status(cudaGetLastError());
}

using PairConv = PairCfg<3, 3, true, true>;    // int8 weights, CTA pair, 64-K fp16 stages
using PairConvWide = PairCfg<2, 2, true, true, 2, true>;  // the same with 128-K fp16 stages
using PairWide = PairCfg<4, 4, true, false>;   // pre-widened weights, CTA pair
using PairWideW = PairCfg<4, 2, true, false, 2, true>;  // the same with 128-K fp16 stages
using CfgConv128 = GemmCfg<128, 3, 3, true, true>;   // int8 weights
using CfgWide128 = GemmCfg<128, 4, 4, true, false>;  // weights pre-widened to fp16 codes
using CfgConv256 = GemmCfg<256, 2, 2, true, true>;
using CfgWide256 = GemmCfg<256, 3, 3, true, false>;

// The int8-code pair kernel stages 128 K of fp16 codes per hand-off unless the
// option asks for 64 or the fp32 chunk is not a whole number of 128-K stages.
bool pair_wide_stages() { return g_opt.pair_stage_k != 64 && g_opt.chunk_k % 128 == 0; }


int conv_pair_clusters(DeviceInfo* d) {
  return pair_wide_stages() ? pair_cluster_capacity<PairConvWide>(d, 2)
                            : pair_cluster_capacity<PairConv>(d, 0);
}
int wide_pair_clusters(DeviceInfo* d) {
  return pair_wide_stages() ? pair_cluster_capacity<PairWideW>(d, 3)
                            : pair_cluster_capacity<PairWide>(d, 1);
}

// Common GEMM driver.  b16 = weights given as fp16 codes instead of int8.
// ws_cap bounds the workspace the plan may ask for (the no-alloc entry's
// fixed array); the plan falls back from stream-K when that is too small.
i8_status gemm_common(const int8_t* aq, const void* wb, bool b16, int64_t M, int64_t N, int64_t K,
                      int out_mode, void* out, int64_t ldo, const float* s_a, const float* s_w,
                      const void* bias, void* ws, size_t ws_bytes, cudaStream_t st,
                      size_t ws_cap = SIZE_MAX) {
  if (M < 0 || N < 0 || K <= 0) return I8_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > 131072 || M > INT32_MAX || N > INT32_MAX) return I8_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return I8_OK;
  if (!aq || !wb || !out || ldo < N) return I8_ERR_INVALID_ARG;
  if (out_mode == kOutBf16 && (!s_a || !s_w)) return I8_ERR_INVALID_ARG;
  if (!aligned16(aq) || !aligned16(wb) || !aligned16(out)) return I8_ERR_ALIGNMENT;
  if (out_mode == kOutBf16 && (ldo % 8 != 0 || !aligned4(s_a) || !aligned16(s_w) ||
                               (bias && !aligned16(bias))))
    return I8_ERR_ALIGNMENT;
  if (out_mode == kOutInt32 && ldo % 4 != 0) return I8_ERR_ALIGNMENT;
  DeviceInfo* d;
  if (i8_status e = device_info(&d, nullptr)) return e;
  const int clusters = b16 ? wide_pair_clusters(d)
                           : conv_pair_clusters(d);
  const Plan pl = make_plan(M, N, K, d->sms, clusters, b16, ws_cap, skinny_fit(d, b16, M));
  if (pl.ws_bytes > 0) {
    if (!ws || ws_bytes < pl.ws_bytes) return I8_ERR_WORKSPACE;
    if (!aligned16(ws)) return I8_ERR_ALIGNMENT;
  }
  if (pl.skinny)
    return b16 ? skinny_route<kSkW16>(d, pl, aq, wb, M, N, K, out_mode, out, ldo, s_a, s_w, bias, st)
               : skinny_route<kSkI8>(d, pl, aq, wb, M, N, K, out_mode, out, ldo, s_a, s_w, bias, st);
  CUtensorMap ma, mb;
  const uint32_t bn = pl.pair ? 128u : static_cast<uint32_t>(pl.bn);
  if (!encode_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, aq, K, M, K, 128, 128)) return I8_ERR_CUDA;
  if (b16) {
    if (!encode_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, wb, K, N, 2 * K, 64, bn))
      return I8_ERR_CUDA;
  } else {
    if (!encode_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, wb, K, N, K, 128, bn)) return I8_ERR_CUDA;
  }
  GemmParams gp{};
  gp.M = static_cast<int>(M);
  gp.N = static_cast<int>(N);
  gp.K = static_cast<int>(K);
  gp.num_m_blk = pl.num_m;
  gp.num_n_blk = pl.num_n;
  gp.n_fastest = pl.n_fastest;
  gp.splits = pl.splits;
  gp.kb_per_split = pl.kb_per_split;
  gp.total_kb = pl.total_kb;
  gp.num_tiles = pl.num_tiles;
  gp.chunk_stages = pl.chunk_stages;
  gp.s_a = s_a;
  gp.s_w = s_w;
  gp.bias = static_cast<const uint16_t*>(bias);
  if (pl.splits > 1) {
    gp.out_mode = kOutPartial;
    gp.out = ws;
    gp.ldo = pl.ws_ld;
    gp.split_stride = static_cast<int64_t>(M) * pl.ws_ld;
  } else {
    gp.out_mode = out_mode;
    gp.out = out;
    gp.ldo = ldo;
    gp.split_stride = 0;
  }
  CUtensorMap my;
  if (!encode_out(&my, gp.out_mode == kOutBf16, gp.out, static_cast<uint64_t>(N),
                  static_cast<uint64_t>(M), static_cast<uint64_t>(gp.ldo),
                  static_cast<uint64_t>(pl.splits)))
    return I8_ERR_CUDA;
  // Stream-K partial slots: {256 columns, 256 rows, 1 per sharing pair} int32.
  CUtensorMap mp = my;
  if (pl.stream_k) {
    gp.stream_k = 1;
    gp.sk_waves = pl.sk_waves;
    gp.sk_pairs = pl.sk_pairs;
    gp.sk_arrive = static_cast<unsigned long long*>(ws);
    gp.sk_part = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(ws) + pl.sk_arrive_bytes);
    gp.sk_epoch = next_sk_epoch();
    if (!encode_out(&mp, false, gp.sk_part, 256, 256, 256, static_cast<uint64_t>(pl.sk_pairs)))
      return I8_ERR_CUDA;
  }
  i8_status e;
  if (pl.pair) {
    e = b16 ? (pair_wide_stages() ? launch_pair_cfg<PairWideW>(ma, mb, my, mp, gp, pl.grid, st)
                                  : launch_pair_cfg<PairWide>(ma, mb, my, mp, gp, pl.grid, st))
            : (pair_wide_stages() ? launch_pair_cfg<PairConvWide>(ma, mb, my, mp, gp, pl.grid, st)
                                  : launch_pair_cfg<PairConv>(ma, mb, my, mp, gp, pl.grid, st));
  } else if (pl.bn == 256) {
    e = b16 ? launch_gemm_cfg<CfgWide256>(d, 3, ma, mb, my, gp, pl.grid, st)
            : launch_gemm_cfg<CfgConv256>(d, 2, ma, mb, my, gp, pl.grid, st);
  } else {
    e = b16 ? launch_gemm_cfg<CfgWide128>(d, 1, ma, mb, my, gp, pl.grid, st)
            : launch_gemm_cfg<CfgConv128>(d, 0, ma, mb, my, gp, pl.grid, st);
  }
  if (e != I8_OK) return e;
  if (pl.splits > 1) {
    GemmParams rp = gp;
    rp.out_mode = out_mode;
    rp.out = out;
    rp.ldo = ldo;
    const int64_t groups = M * ((N + 3) / 4);
    const int64_t blocks = std::min<int64_t>((groups + 255) / 256, static_cast<int64_t>(d->sms) * 16);
    return cuda_status(launch_pdl(splitk_reduce_kernel, dim3(static_cast<unsigned>(blocks)),
                                  dim3(256), 0, st, static_cast<const int32_t*>(ws),
                                  gp.split_stride, pl.ws_ld, pl.splits, rp));
  }
  return I8_OK;
}

// ----------------------------------------------------------------- direct (converter-free) GEMM
template <int KIND>
int direct_cluster_capacity(DeviceInfo* d) {
  static int cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return d->sms / 2;
  if (cached[dev] > 0) return cached[dev];
  using Cfg = DirectCfg<KIND>;
  auto kern = gemm_direct_pair_kernel<KIND>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (d->sms / 2), 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  if (n <= 0) n = d->sms / 2;
  cached[dev] = n;
  return n;
}

// Plan of the direct GEMM: 256 x 256 tiles of 128-byte-deep K blocks (128
// E4M3 or 64 fp16 codes); when the tiles leave CTA pairs idle, K splits of
// at least 4 blocks by the same wave-efficiency rule as the int8 table.
// ws: 4-byte partials (fp32 or int32) [splits][M][round_up(N, 4)].
struct DirectPlan {
  int num_m, num_n, total_kb, splits, kb_per_split;
  int64_t tiles;
  int64_t ldw;
  size_t ws_bytes;
};

// Modelled time (us) of a direct-kernel plan with `splits` K splits, up to a
// start-up cost common to every plan.  Grid fill alone favours many short
// items, but an item cannot retire faster than its epilogue (the accumulator
// is double-buffered, so an item's epilogue overlaps the next item's MMAs),
// and a split plan writes and re-reads fp32/int32 partial planes.  Per CTA
// pair on GB300: a 256 x 256 tile advances one 128-byte K block in 0.31 us
// (either kind); an epilogue takes 2 us for bf16 and 3 us for a 4-byte
// partial; the fix-up costs 2 us plus 8 bytes per partial element at 15 TB/s
// while the planes fit in L2 (64 MB), else at 6.5 TB/s.  The constants were
// fitted to timings of both kinds over the DiT layer shapes.
double direct_plan_us(int64_t tiles, int pairs, int total_kb, int splits, int64_t M, int64_t N) {
  const int kbps = (total_kb + splits - 1) / splits;
  const int s = (total_kb + kbps - 1) / kbps;
  const int64_t rounds = (tiles * s + pairs - 1) / pairs;
  const double t_epi = s > 1 ? 3.0 : 2.0;
  double t = static_cast<double>(rounds) * std::max(0.31 * kbps, t_epi) + t_epi;
  if (s > 1) {
    const double bytes = 8.0 * s * static_cast<double>(M) * static_cast<double>(N);
    t += 2.0 + bytes / (bytes <= 128.0 * (1 << 20) ? 15e6 : 6.5e6);
  }
  return t;
}

DirectPlan plan_direct(int64_t M, int64_t N, int64_t K, int pairs, int bk) {
  DirectPlan p{};
  p.num_m = static_cast<int>((M + 255) / 256);
  p.num_n = static_cast<int>((N + 255) / 256);
  p.total_kb = static_cast<int>((K + bk - 1) / bk);
  p.tiles = static_cast<int64_t>(p.num_m) * p.num_n;
  // splits: the cheapest plan under direct_plan_us, only when the tiles
  // leave pairs idle, and never below four K blocks per split
  p.splits = 1;
  if (p.tiles < pairs) {
    double best = direct_plan_us(p.tiles, pairs, p.total_kb, 1, M, N);
    const int max_s = std::max(1, std::min(16, p.total_kb / 4));
    for (int s = 2; s <= max_s; ++s) {
      const double t = direct_plan_us(p.tiles, pairs, p.total_kb, s, M, N);
      if (t < best - 1e-9) {
        best = t;
        p.splits = s;
      }
    }
  }
  if (g_opt.force_splits > 0) p.splits = std::min(g_opt.force_splits, p.total_kb);
  p.kb_per_split = (p.total_kb + p.splits - 1) / p.splits;
  p.splits = (p.total_kb + p.kb_per_split - 1) / p.kb_per_split;
  p.ldw = (N + 3) / 4 * 4;
  p.ws_bytes = p.splits > 1 ? static_cast<size_t>(p.splits) * static_cast<size_t>(M) *
                                  static_cast<size_t>(p.ldw) * 4
                            : 0;
  return p;
}

// The direct GEMM: E4M3 codes (KIND = kDirectE4M3) or fp16 values of int8
// codes (kDirectF16) in; bf16 (dequant + bias) or the raw accumulator (fp32
// for E4M3, exact int32 for fp16 codes) out.  One persistent launch of the
// pair kernel, plus the split-K fix-up when the plan splits K; rows and
// columns beyond M, N are zero-filled on load and clipped on store.
template <int KIND>
i8_status gemm_direct_common(const void* aq, const void* wq, int64_t M, int64_t N, int64_t K,
                             int out_mode, void* out, int64_t ldo, const float* s_a,
                             const float* s_w, const void* bias, void* ws, size_t ws_bytes,
                             cudaStream_t st) {
  using Cfg = DirectCfg<KIND>;
  if (M < 0 || N < 0 || K <= 0) return I8_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > 131072 || M > INT32_MAX || N > INT32_MAX) return I8_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return I8_OK;
  if (!aq || !wq || !out || ldo < N) return I8_ERR_INVALID_ARG;
  if (out_mode == kOutBf16 && (!s_a || !s_w)) return I8_ERR_INVALID_ARG;
  if (!aligned16(aq) || !aligned16(wq) || !aligned16(out)) return I8_ERR_ALIGNMENT;
  if (out_mode == kOutBf16 && (ldo % 8 != 0 || !aligned4(s_a) || !aligned16(s_w) ||
                               (bias && !aligned16(bias))))
    return I8_ERR_ALIGNMENT;
  if (out_mode != kOutBf16 && ldo % 4 != 0) return I8_ERR_ALIGNMENT;
  DeviceInfo* d;
  if (i8_status e = device_info(&d, nullptr)) return e;
  if (M <= g_opt.skinny_max_m) {
    // few tokens: the weight-streaming kernel, no workspace
    constexpr int SK = KIND == kDirectF16 ? kSkF16 : kSkE4M3;
    Plan sp;
    plan_skinny(sp, M, N, K, d->sms, skinny_fit_k<SK>(d, M));
    return skinny_route<SK>(d, sp, aq, wq, M, N, K, out_mode, out, ldo, s_a, s_w, bias, st);
  }
  const int clusters = direct_cluster_capacity<KIND>(d);
  const DirectPlan pl = plan_direct(M, N, K, clusters, Cfg::BK);
  if (pl.tiles * pl.splits > INT32_MAX) return I8_ERR_UNSUPPORTED;
  if (pl.ws_bytes > 0) {
    if (!ws || ws_bytes < pl.ws_bytes) return I8_ERR_WORKSPACE;
    if (!aligned16(ws)) return I8_ERR_ALIGNMENT;
  }
  CUtensorMap ma, mb, my;
  const CUtensorMapDataType dt =
      KIND == kDirectF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint64_t row_bytes = KIND == kDirectF16 ? 2 * K : K;
  if (!encode_2d(&ma, dt, aq, K, M, row_bytes, Cfg::BK, Cfg::BM) ||
      !encode_2d(&mb, dt, wq, K, N, row_bytes, Cfg::BK, Cfg::BN))
    return I8_ERR_CUDA;
  GemmParams gp{};
  gp.M = static_cast<int>(M);
  gp.N = static_cast<int>(N);
  gp.K = static_cast<int>(K);
  gp.num_m_blk = pl.num_m;
  gp.num_n_blk = pl.num_n;
  gp.n_fastest = tile_order_n_fastest(M, N);
  gp.splits = pl.splits;
  gp.total_kb = pl.total_kb;
  gp.kb_per_split = pl.kb_per_split;
  gp.num_tiles = static_cast<int>(pl.tiles);
  gp.chunk_stages = g_opt.chunk_k / 64;   // fp16 codes: 64 K per block
  gp.s_a = s_a;
  gp.s_w = s_w;
  gp.bias = static_cast<const uint16_t*>(bias);
  if (pl.splits > 1) {
    gp.out_mode = kOutPartial;
    gp.out = ws;
    gp.ldo = pl.ldw;
    gp.split_stride = M * pl.ldw;
    if (!encode_out(&my, false, ws, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                    static_cast<uint64_t>(pl.ldw), static_cast<uint64_t>(pl.splits)))
      return I8_ERR_CUDA;
  } else {
    gp.out_mode = out_mode;
    gp.out = out;
    gp.ldo = ldo;
    if (!encode_out(&my, out_mode == kOutBf16, out, static_cast<uint64_t>(N),
                    static_cast<uint64_t>(M), static_cast<uint64_t>(ldo), 1))
      return I8_ERR_CUDA;
  }
  const int grid = 2 * static_cast<int>(std::min<int64_t>(clusters, pl.tiles * pl.splits));
  if (cudaError_t e = launch_pdl(gemm_direct_pair_kernel<KIND>, dim3(grid), dim3(Cfg::THREADS),
                                 Cfg::SMEM_BYTES, st, ma, mb, my, gp))
    return cuda_status(e);
  if (pl.splits > 1) {
    GemmParams rp = gp;
    rp.out_mode = out_mode;
    rp.out = out;
    rp.ldo = ldo;
    const int64_t groups = M * ((N + 3) / 4);
    const int64_t blocks = std::min<int64_t>((groups + 255) / 256, static_cast<int64_t>(d->sms) * 16);
    if (KIND == kDirectF16)
      return cuda_status(launch_pdl(splitk_reduce_kernel, dim3(static_cast<unsigned>(blocks)),
                                    dim3(256), 0, st, static_cast<const int32_t*>(ws),
                                    gp.split_stride, pl.ldw, pl.splits, rp));
    return cuda_status(launch_pdl(splitk_reduce_f32_kernel, dim3(static_cast<unsigned>(blocks)),
                                  dim3(256), 0, st, static_cast<const float*>(ws),
                                  gp.split_stride, pl.ldw, pl.splits, rp));
  }
  return I8_OK;
}

// ----------------------------------------------------------------- no-alloc variant
// Split-K scratch for i8_gemm_dequant_bias_bf16_noalloc: a fixed array in the
// library's own device memory, so that entry point never allocates.  Every
// GPU that loads the library holds these bytes until the process exits.
constexpr size_t kStaticWsBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// Device address of g_static_ws per device.  In host code the symbol is only
// a host-side stand-in, so the address is looked up once per device (with
// that device current) and cached.
void* g_static_ws_ptr[kMaxDevices] = {};

i8_status static_ws_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return I8_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_static_ws_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return I8_ERR_CUDA;
    g_static_ws_ptr[dev] = p;
  }
  *out = g_static_ws_ptr[dev];
  return I8_OK;
}

}  // namespace
}  // namespace i8

using namespace i8;

extern "C" {

const char* i8_status_string(i8_status s) {
  switch (s) {
    case I8_OK: return "I8_OK";
    case I8_ERR_INVALID_ARG: return "I8_ERR_INVALID_ARG";
    case I8_ERR_ALIGNMENT: return "I8_ERR_ALIGNMENT";
    case I8_ERR_UNSUPPORTED: return "I8_ERR_UNSUPPORTED";
    case I8_ERR_WORKSPACE: return "I8_ERR_WORKSPACE";
    case I8_ERR_CUDA: return "I8_ERR_CUDA";
    case I8_ERR_DEVICE_TIMEOUT: return "I8_ERR_DEVICE_TIMEOUT";
  }
  return "I8_ERR_UNKNOWN";
}

const char* i8_version(void) { return "i8 0.1.0 sm_103a"; }

i8_status i8_quant_weight_perchannel(const void* w, int64_t N, int64_t K, int64_t ldw, int8_t* wq,
                                     int64_t ldq, float* s_w, i8_stream_t stream) {
  I8_NVTX();
  return quant_rows(w, N, K, ldw, wq, ldq, s_w, reinterpret_cast<cudaStream_t>(stream));
}

i8_status i8_quant_act_pertoken(const void* x, int64_t M, int64_t K, int64_t ldx, int8_t* aq,
                                int64_t ldq, float* s_a, i8_stream_t stream) {
  I8_NVTX();
  return quant_rows(x, M, K, ldx, aq, ldq, s_a, reinterpret_cast<cudaStream_t>(stream));
}

i8_status i8_quant_weight_perchannel_e4m3(const void* w, int64_t N, int64_t K, int64_t ldw,
                                          uint8_t* wq, int64_t ldq, float* s_w,
                                          i8_stream_t stream) {
  I8_NVTX();
  return quant_rows(w, N, K, ldw, reinterpret_cast<int8_t*>(wq), ldq, s_w,
                    reinterpret_cast<cudaStream_t>(stream), kQuantE4M3);
}

i8_status i8_quant_act_pertoken_e4m3(const void* x, int64_t M, int64_t K, int64_t ldx,
                                     uint8_t* aq, int64_t ldq, float* s_a, i8_stream_t stream) {
  I8_NVTX();
  return quant_rows(x, M, K, ldx, reinterpret_cast<int8_t*>(aq), ldq, s_a,
                    reinterpret_cast<cudaStream_t>(stream), kQuantE4M3);
}

size_t i8_gemm_e4m3_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  I8_NVTX();
  if (M <= 0 || N <= 0 || K <= 0 || K % 16 != 0 || K > 131072 || M > INT32_MAX || N > INT32_MAX)
    return 0;
  if (M <= g_opt.skinny_max_m) return 0;   // the weight-streaming kernel needs none
  DeviceInfo* d;
  if (device_info(&d, nullptr) != I8_OK) return 0;
  return plan_direct(M, N, K, direct_cluster_capacity<kDirectE4M3>(d),
                     DirectCfg<kDirectE4M3>::BK).ws_bytes;
}

i8_status i8_gemm_e4m3_f32(const uint8_t* aq, const uint8_t* wq, int64_t M, int64_t N, int64_t K,
                           float* c, int64_t ldc, void* ws, size_t ws_bytes,
                           i8_stream_t stream) {
  I8_NVTX();
  return gemm_direct_common<kDirectE4M3>(aq, wq, M, N, K, kOutInt32, c, ldc, nullptr, nullptr,
                                         nullptr, ws, ws_bytes,
                                         reinterpret_cast<cudaStream_t>(stream));
}

i8_status i8_gemm_e4m3_dequant_bias_bf16(const uint8_t* aq, const float* s_a, const uint8_t* wq,
                                         const float* s_w, const void* bias, int64_t M,
                                         int64_t N, int64_t K, void* y, int64_t ldy, void* ws,
                                         size_t ws_bytes, i8_stream_t stream) {
  I8_NVTX();
  return gemm_direct_common<kDirectE4M3>(aq, wq, M, N, K, kOutBf16, y, ldy, s_a, s_w, bias, ws,
                                         ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

i8_status i8_quant_act_pertoken_f16codes(const void* x, int64_t M, int64_t K, int64_t ldx,
                                         void* q16, int64_t ldq, float* s_a,
                                         i8_stream_t stream) {
  I8_NVTX();
  return quant_rows(x, M, K, ldx, static_cast<int8_t*>(q16), ldq, s_a,
                    reinterpret_cast<cudaStream_t>(stream), kQuantF16);
}

size_t i8_gemm_f16codes_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  I8_NVTX();
  if (M <= 0 || N <= 0 || K <= 0 || K % 16 != 0 || K > 131072 || M > INT32_MAX || N > INT32_MAX)
    return 0;
  if (M <= g_opt.skinny_max_m) return 0;   // the weight-streaming kernel needs none
  DeviceInfo* d;
  if (device_info(&d, nullptr) != I8_OK) return 0;
  return plan_direct(M, N, K, direct_cluster_capacity<kDirectF16>(d),
                     DirectCfg<kDirectF16>::BK).ws_bytes;
}

i8_status i8_gemm_int32_f16codes(const void* a16, const void* w16, int64_t M, int64_t N,
                                 int64_t K, int32_t* c, int64_t ldc, void* ws, size_t ws_bytes,
                                 i8_stream_t stream) {
  I8_NVTX();
  return gemm_direct_common<kDirectF16>(a16, w16, M, N, K, kOutInt32, c, ldc, nullptr, nullptr,
                                        nullptr, ws, ws_bytes,
                                        reinterpret_cast<cudaStream_t>(stream));
}

i8_status i8_gemm_dequant_bias_bf16_f16codes(const void* a16, const float* s_a, const void* w16,
                                             const float* s_w, const void* bias, int64_t M,
                                             int64_t N, int64_t K, void* y, int64_t ldy,
                                             void* ws, size_t ws_bytes, i8_stream_t stream) {
  I8_NVTX();
  return gemm_direct_common<kDirectF16>(a16, w16, M, N, K, kOutBf16, y, ldy, s_a, s_w, bias, ws,
                                        ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

i8_status i8_layernorm_quant_act_pertoken(const void* h, int64_t M, int64_t K, int64_t ldh,
                                          float eps, int fmt, void* q, int64_t ldq, float* s_a,
                                          void* y, int64_t ldy, i8_stream_t stream) {
  I8_NVTX();
  return producer_quant(kOpLayerNorm, h, M, K, ldh, eps, fmt, q, ldq, s_a, y, ldy,
                        reinterpret_cast<cudaStream_t>(stream));
}

i8_status i8_gelu_quant_act_pertoken(const void* u, int64_t M, int64_t K, int64_t ldu, int fmt,
                                     void* q, int64_t ldq, float* s_a, void* y, int64_t ldy,
                                     i8_stream_t stream) {
  I8_NVTX();
  return producer_quant(kOpGelu, u, M, K, ldu, 0.0f, fmt, q, ldq, s_a, y, ldy,
                        reinterpret_cast<cudaStream_t>(stream));
}

size_t i8_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  I8_NVTX();
  if (M <= 0 || N <= 0 || K <= 0 || K % 16 != 0 || K > 131072 || M > INT32_MAX || N > INT32_MAX)
    return 0;
  DeviceInfo* d;
  if (device_info(&d, nullptr) != I8_OK) return 0;
  // the larger of the two weight formats' plans, so one query serves both
  const size_t a = make_plan(M, N, K, d->sms, conv_pair_clusters(d), false,
                             SIZE_MAX, skinny_fit(d, false, M)).ws_bytes;
  const size_t b = make_plan(M, N, K, d->sms, wide_pair_clusters(d), true,
                             SIZE_MAX, skinny_fit(d, true, M)).ws_bytes;
  return a > b ? a : b;
}

i8_status i8_gemm_int32(const int8_t* aq, const int8_t* wq, int64_t M, int64_t N, int64_t K,
                        int32_t* c, int64_t ldc, void* ws, size_t ws_bytes, i8_stream_t stream) {
  I8_NVTX();
  return gemm_common(aq, wq, false, M, N, K, kOutInt32, c, ldc, nullptr, nullptr, nullptr, ws,
                     ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

i8_status i8_gemm_dequant_bias_bf16(const int8_t* aq, const float* s_a, const int8_t* wq,
                                    const float* s_w, const void* bias, int64_t M, int64_t N,
                                    int64_t K, void* y, int64_t ldy, void* ws, size_t ws_bytes,
                                    i8_stream_t stream) {
  I8_NVTX();
  return gemm_common(aq, wq, false, M, N, K, kOutBf16, y, ldy, s_a, s_w, bias, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

i8_status i8_gemm_dequant_bias_bf16_noalloc(const int8_t* aq, const float* s_a, const int8_t* wq,
                                            const float* s_w, const void* bias, int64_t M,
                                            int64_t N, int64_t K, void* y, int64_t ldy,
                                            i8_stream_t stream) {
  I8_NVTX();
  // Same checks and kernels as i8_gemm_dequant_bias_bf16; only the split-K
  // scratch comes from the library's fixed device array, and the plan is
  // capped to its size (fewer K splits, or none).  What the array must hold
  // at the start of a call: the tiled kernels' split-K partials are written
  // in full before the reduction reads them; the few-token kernel uses none
  // of it (its K splits meet in distributed shared memory); the stream-K
  // arrival words carry a per-launch epoch tag, so words left by an earlier
  // call count as zero.
  void* ws = nullptr;
  if (M > 0 && N > 0 && K > 0 && K % 16 == 0 && K <= 131072 && M <= INT32_MAX &&
      N <= INT32_MAX) {
    DeviceInfo* d;
    if (i8_status e = device_info(&d, nullptr)) return e;
    if (make_plan(M, N, K, d->sms, conv_pair_clusters(d), false, kStaticWsBytes,
                  skinny_fit(d, false, M))
            .ws_bytes > kStaticWsBytes)
      return I8_ERR_WORKSPACE;
    if (i8_status e = static_ws_address(&ws)) return e;
  }
  return gemm_common(aq, wq, false, M, N, K, kOutBf16, y, ldy, s_a, s_w, bias, ws,
                     ws ? kStaticWsBytes : 0, reinterpret_cast<cudaStream_t>(stream),
                     kStaticWsBytes);
}

i8_status i8_widen_weight_codes(const int8_t* wq, int64_t N, int64_t K, void* w16,
                                i8_stream_t stream) {
  I8_NVTX();
  if (N < 0 || K <= 0) return I8_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > 131072) return I8_ERR_UNSUPPORTED;
  if (N == 0) return I8_OK;
  if (!wq || !w16) return I8_ERR_INVALID_ARG;
  if (!aligned16(wq) || !aligned16(w16)) return I8_ERR_ALIGNMENT;
  DeviceInfo* d;
  if (i8_status e = device_info(&d, nullptr)) return e;
  const int64_t n16 = N * K / 16;
  const int64_t blocks = std::min<int64_t>((n16 + 255) / 256, static_cast<int64_t>(d->sms) * 8);
  widen_codes_kernel<<<static_cast<unsigned>(blocks), 256, 0,
                       reinterpret_cast<cudaStream_t>(stream)>>>(wq, static_cast<uint16_t*>(w16),
                                                                 n16);
  return cuda_status(cudaGetLastError());
}

i8_status i8_gemm_dequant_bias_bf16_w16(const int8_t* aq, const float* s_a, const void* w16,
                                        const float* s_w, const void* bias, int64_t M, int64_t N,
                                        int64_t K, void* y, int64_t ldy, void* ws,
                                        size_t ws_bytes, i8_stream_t stream) {
  I8_NVTX();
  return gemm_common(aq, w16, true, M, N, K, kOutBf16, y, ldy, s_a, s_w, bias, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

i8_status i8_set_option(i8_option opt, int64_t value) {
  switch (opt) {
    case I8_OPT_CHUNK_K:
      if (value < 64 || value > 1024 || value % 64 != 0) return I8_ERR_INVALID_ARG;
      g_opt.chunk_k = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_FORCE_SPLITS:
      if (value < 0 || value > 1024) return I8_ERR_INVALID_ARG;
      g_opt.force_splits = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_MAX_CTAS:
      if (value < 0) return I8_ERR_INVALID_ARG;
      g_opt.max_ctas = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_QUANT_VPL:
      if (value < 1 || value > 16) return I8_ERR_INVALID_ARG;
      g_opt.quant_vpl = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_CTA_PAIR:
      if (value < 0 || value > 2) return I8_ERR_INVALID_ARG;
      g_opt.cta_pair = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_SKINNY_MAX_M:
      if (value < 0 || value > 16) return I8_ERR_INVALID_ARG;
      g_opt.skinny_max_m = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_PDL:
      if (value != 0 && value != 1) return I8_ERR_INVALID_ARG;
      g_opt.pdl = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_STREAM_K:
      if (value < 0 || value > 2) return I8_ERR_INVALID_ARG;
      g_opt.stream_k = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_QUANT_ROWS:
      if (value < 0 || value > 8) return I8_ERR_INVALID_ARG;
      g_opt.quant_rows = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_TILE_N:
      if (value != 0 && value != 128 && value != 256) return I8_ERR_INVALID_ARG;
      g_opt.force_bn = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_NVTX:
      if (value != 0 && value != 1) return I8_ERR_INVALID_ARG;
      g_opt.nvtx = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_PAIR_STAGE_K:
      if (value != 0 && value != 64 && value != 128) return I8_ERR_INVALID_ARG;
      g_opt.pair_stage_k = static_cast<int>(value);
      return I8_OK;
    case I8_OPT_RASTER:
      if (value < 0 || value > 2) return I8_ERR_INVALID_ARG;
      g_opt.raster = static_cast<int>(value);
      return I8_OK;
  }
  return I8_ERR_INVALID_ARG;
}

i8_status i8_get_option(i8_option opt, int64_t* value) {
  if (!value) return I8_ERR_INVALID_ARG;
  switch (opt) {
    case I8_OPT_CHUNK_K: *value = g_opt.chunk_k; return I8_OK;
    case I8_OPT_FORCE_SPLITS: *value = g_opt.force_splits; return I8_OK;
    case I8_OPT_MAX_CTAS: *value = g_opt.max_ctas; return I8_OK;
    case I8_OPT_TILE_N: *value = g_opt.force_bn; return I8_OK;
    case I8_OPT_QUANT_VPL: *value = g_opt.quant_vpl; return I8_OK;
    case I8_OPT_CTA_PAIR: *value = g_opt.cta_pair; return I8_OK;
    case I8_OPT_SKINNY_MAX_M: *value = g_opt.skinny_max_m; return I8_OK;
    case I8_OPT_PDL: *value = g_opt.pdl; return I8_OK;
    case I8_OPT_QUANT_ROWS: *value = g_opt.quant_rows; return I8_OK;
    case I8_OPT_STREAM_K: *value = g_opt.stream_k; return I8_OK;
    case I8_OPT_NVTX: *value = g_opt.nvtx; return I8_OK;
    case I8_OPT_PAIR_STAGE_K: *value = g_opt.pair_stage_k; return I8_OK;
    case I8_OPT_RASTER: *value = g_opt.raster; return I8_OK;
  }
  return I8_ERR_INVALID_ARG;
}

// The same planners the GEMM calls run (make_plan, plan_direct), fed either
// the caller's machine figures or the current device's.
i8_status i8_plan_query(int64_t M, int64_t N, int64_t K, i8_route route, int sms, int pairs,
                        int skinny_slots_in, size_t ws_cap, i8_plan_info* out) {
  if (!out || M <= 0 || N <= 0 || K <= 0 || sms < 0 || pairs < 0 || skinny_slots_in < 0)
    return I8_ERR_INVALID_ARG;
  if (route != I8_ROUTE_INT8 && route != I8_ROUTE_W16 && route != I8_ROUTE_F16CODES &&
      route != I8_ROUTE_E4M3)
    return I8_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > 131072 || M > INT32_MAX || N > INT32_MAX) return I8_ERR_UNSUPPORTED;
  const bool b16 = route == I8_ROUTE_W16;
  // a machine described by hand: clusters assumed to pack the slots fully
  SkinnyFit fit;
  fit.slots = skinny_slots_in;
  if (sms == 0) {
    DeviceInfo* d;
    if (i8_status e = device_info(&d, nullptr)) return e;
    sms = d->sms;
    pairs = route == I8_ROUTE_E4M3       ? direct_cluster_capacity<kDirectE4M3>(d)
            : route == I8_ROUTE_F16CODES ? direct_cluster_capacity<kDirectF16>(d)
            : b16                        ? wide_pair_clusters(d)
                                         : conv_pair_clusters(d);
    fit = route == I8_ROUTE_E4M3       ? skinny_fit_k<kSkE4M3>(d, M)
          : route == I8_ROUTE_F16CODES ? skinny_fit_k<kSkF16>(d, M)
                                       : skinny_fit(d, b16, M);
  }
  if (fit.slots <= 0) fit.slots = 2 * sms;
  if (pairs == 0) pairs = std::max(1, sms / 2);
  i8_plan_info r{};
  r.n_fastest = tile_order_n_fastest(M, N);
  const bool direct_route = route == I8_ROUTE_F16CODES || route == I8_ROUTE_E4M3;
  if (direct_route && M <= g_opt.skinny_max_m) {
    // few tokens: the weight-streaming kernel, as on the int8 routes
    Plan pl;
    plan_skinny(pl, M, N, K, sms, fit);
    r.kernel = I8_KERNEL_SKINNY;
    r.tile_m = static_cast<int>(M);
    r.tile_n = kSkinnyRows;
    r.num_m = 1;
    r.num_n = pl.num_n;
    r.block_k = kSkinnyK;
    r.total_kb = pl.total_kb;
    r.splits = pl.splits;
    r.kb_per_split = pl.kb_per_split;
    r.grid = pl.grid;
    r.ws_bytes = 0;
  } else if (direct_route) {
    const int bk = route == I8_ROUTE_E4M3 ? DirectCfg<kDirectE4M3>::BK : DirectCfg<kDirectF16>::BK;
    const DirectPlan pl = plan_direct(M, N, K, pairs, bk);
    if (pl.tiles * pl.splits > INT32_MAX) return I8_ERR_UNSUPPORTED;
    r.kernel = I8_KERNEL_DIRECT;
    r.tile_m = r.tile_n = 256;
    r.num_m = pl.num_m;
    r.num_n = pl.num_n;
    r.block_k = bk;
    r.total_kb = pl.total_kb;
    r.splits = pl.splits;
    r.kb_per_split = pl.kb_per_split;
    r.grid = 2 * static_cast<int>(std::min<int64_t>(pairs, pl.tiles * pl.splits));
    r.ws_bytes = static_cast<int64_t>(pl.ws_bytes);
    r.model_us = direct_plan_us(pl.tiles, pairs, pl.total_kb, pl.splits, M, N);
  } else {
    const Plan pl = make_plan(M, N, K, sms, pairs, b16, ws_cap ? ws_cap : SIZE_MAX,
                              fit);
    r.num_m = pl.num_m;
    r.num_n = pl.num_n;
    r.total_kb = pl.total_kb;
    r.splits = pl.splits;
    r.kb_per_split = pl.kb_per_split;
    r.ws_bytes = static_cast<int64_t>(pl.ws_bytes);
    r.n_fastest = pl.n_fastest;
    r.sk_waves = pl.sk_waves;
    r.sk_pairs = pl.sk_pairs;
    if (pl.skinny) {
      r.kernel = I8_KERNEL_SKINNY;
      r.tile_m = static_cast<int>(M);
      r.tile_n = kSkinnyRows;
      r.block_k = kSkinnyK;
      r.grid = pl.num_n * pl.splits;
    } else {
      r.kernel = pl.stream_k ? I8_KERNEL_PAIR_STREAM_K : pl.pair ? I8_KERNEL_PAIR : I8_KERNEL_TILE;
      r.tile_m = pl.pair ? 256 : 128;
      r.tile_n = pl.bn;
      r.block_k = 128;
      r.grid = pl.grid;
    }
  }
  *out = r;
  return I8_OK;
}

i8_status i8_selftest_timeout(int limit_ms, i8_stream_t stream) {
  I8_NVTX();
  if (limit_ms < 1 || limit_ms > 5000) return I8_ERR_INVALID_ARG;
  selftest_timeout_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned long long>(limit_ms) * 1000000ull);
  return cuda_status(cudaGetLastError());
}

i8_status i8_sync_check(i8_stream_t stream) {
  I8_NVTX();
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return I8_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_status, sizeof(word)) != cudaSuccess) return I8_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return I8_ERR_CUDA;
    if (word & (1u << I8_ERR_DEVICE_TIMEOUT)) return I8_ERR_DEVICE_TIMEOUT;
    return I8_ERR_CUDA;
  }
  return I8_OK;
}

}  // extern "C"

namespace {

// I8_OPTIONS="name=value,..." applied once when the library is loaded.
struct EnvOptions {
  EnvOptions() {
    const char* env = std::getenv("I8_OPTIONS");
    if (!env) return;
    static const struct {
      const char* name;
      i8_option opt;
    } kNames[] = {{"chunk_k", I8_OPT_CHUNK_K},       {"force_splits", I8_OPT_FORCE_SPLITS},
                  {"max_ctas", I8_OPT_MAX_CTAS},     {"tile_n", I8_OPT_TILE_N},
                  {"quant_vpl", I8_OPT_QUANT_VPL},   {"cta_pair", I8_OPT_CTA_PAIR},
                  {"skinny_max_m", I8_OPT_SKINNY_MAX_M}, {"pdl", I8_OPT_PDL},
                  {"quant_rows", I8_OPT_QUANT_ROWS}, {"stream_k", I8_OPT_STREAM_K},
                  {"nvtx", I8_OPT_NVTX},             {"pair_stage_k", I8_OPT_PAIR_STAGE_K},
                  {"raster", I8_OPT_RASTER}};
    const char* p = env;
    while (*p) {
      const char* end = std::strchr(p, ',');
      const size_t len = end ? static_cast<size_t>(end - p) : std::strlen(p);
      const char* eq = static_cast<const char*>(std::memchr(p, '=', len));
      if (eq) {
        const size_t nlen = static_cast<size_t>(eq - p);
        char* vend = nullptr;
        const long long v = std::strtoll(eq + 1, &vend, 10);
        if (vend == p + len) {
          for (const auto& n : kNames)
            if (std::strlen(n.name) == nlen && std::strncmp(n.name, p, nlen) == 0)
              i8_set_option(n.opt, v);
        }
      }
      if (!end) break;
      p = end + 1;
    }
  }
};
EnvOptions g_env_options;

}  // namespace
