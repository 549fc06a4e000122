// engine_probe.cu -- measurement helper, not part of the W8A8 path: the peak
// rate of this GPU's legacy warp-level tensor MMA for int8 (mma.sync
// m16n8k32 s8 x s8 -> s32) and for fp16 (m16n8k16 f16 x f16 -> f32),
// measured with register-only loops.  On sm_103a the int8 warp MMA is the
// only INT8 tensor-core instruction (tcgen05 has no int8 kind there), so its
// rate is the chip's dense INT8 tensor rate that the fused GEMM is compared
// with.  Built as its own small library (libi8probe.so) so the product
// library carries no benchmark code.
#include <cuda_runtime.h>

#include <cstdint>

namespace {

// Four independent accumulator chains per warp keep the pipe busy; the
// operands are arbitrary register values (the rate does not depend on them).
__global__ void __launch_bounds__(256) mma_s8_loop(int iters, int* sink) {
  const int t = threadIdx.x;
  const int a0 = t, a1 = t * 3, a2 = t ^ 5, a3 = t + 7, b0 = t * 11, b1 = t - 1;
  int c[4][4] = {};
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int s = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) s += c[j][0] ^ c[j][1] ^ c[j][2] ^ c[j][3];
  if (s == 0x7fffffff) sink[0] = s;   // keeps the loop live; never true in practice
}

__global__ void __launch_bounds__(256) mma_f16_loop(int iters, int* sink) {
  const uint32_t t = threadIdx.x;
  const uint32_t a0 = t, a1 = t * 3, a2 = t ^ 5, a3 = t + 7, b0 = t * 11, b1 = t - 1;
  float c[4][4] = {};
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
  if (s == 123456789.0f) sink[0] = 1;
}

}  // namespace

extern "C" {

// Best of `reps` timed launches of each loop (4 CTAs of 256 threads per SM)
// on `stream`, after one untimed launch.  Results in TOPS (int8) and
// TFLOP/s (fp16), 2 operations per multiply-add.  Returns 0 on success, or
// the CUDA error code.  `sink` is a device int the loops may write (never in
// practice).
int i8probe_mma_rates(int reps, int iters, int* sink, double* s8_tops, double* f16_tflops,
                      cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (reps < 1 || iters < 1 || !sink || !s8_tops || !f16_tflops) return -1;
  cudaEvent_t e0, e1;
  if ((e = cudaEventCreate(&e0)) != cudaSuccess) return static_cast<int>(e);
  if ((e = cudaEventCreate(&e1)) != cudaSuccess) return static_cast<int>(e);
  const int blocks = 4 * sms, threads = 256;
  const double warps = blocks * threads / 32.0;
  double best[2] = {0.0, 0.0};
  for (int kind = 0; kind < 2 && e == cudaSuccess; ++kind) {
    for (int r = 0; r <= reps && e == cudaSuccess; ++r) {
      cudaEventRecord(e0, stream);
      if (kind == 0) mma_s8_loop<<<blocks, threads, 0, stream>>>(iters, sink);
      else mma_f16_loop<<<blocks, threads, 0, stream>>>(iters, sink);
      cudaEventRecord(e1, stream);
      e = cudaEventSynchronize(e1);
      float ms = 0.0f;
      if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
      if (e != cudaSuccess || r == 0) continue;    // the first launch is a warm-up
      // m16n8k32 (s8) or m16n8k16 (f16) per instruction, 4 per iteration
      const double k = kind == 0 ? 32.0 : 16.0;
      const double rate = 2.0 * 16 * 8 * k * 4.0 * iters * warps / (ms * 1e-3) / 1e12;
      if (rate > best[kind]) best[kind] = rate;
    }
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  *s8_tops = best[0];
  *f16_tflops = best[1];
  return static_cast<int>(e);
}

}  // extern "C"
