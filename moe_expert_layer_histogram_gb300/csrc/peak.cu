// peak.cu -- dense tensor-core rate of the layer's MMA kinds on this GPU.
//
// The roofline of a block-scaled contraction needs the tensor pipe's own
// rate for that kind, which no library call reports for the FP4 and FP8
// block-scaled kinds.  This kernel measures it: one persistent CTA per SM
// issues back-to-back tcgen05.mma (M = 128, N = 128 or 256) on operands that
// stay resident in shared memory, so no global traffic enters the loop.  The
// operand values are zero; the rate of the tensor pipe does not depend on
// them.  Optionally the loop also re-copies the scale tiles into TMEM
// before every group of four MMAs, exactly as the layer's GEMM does per
// stage, which measures what those copies cost the tensor pipe.
#include <cuda_runtime.h>

#include "internal.h"
#include "moe.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kRateThreads = 128;

__device__ int g_rate_status;

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int FMT, int N, bool COPY_SF>
__global__ void __launch_bounds__(kRateThreads, 1) mma_rate_kernel(int iters) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  constexpr int kA = 128 * 128, kB = N * 128, kSf = 16 * 512;
  uint8_t* a = smem;
  uint8_t* b = smem + kA;
  uint8_t* sf = b + kB;
  uint64_t* done = reinterpret_cast<uint64_t*>(sf + kSf);
  uint32_t* holder = reinterpret_cast<uint32_t*>(done + 1);

  for (int i = threadIdx.x; i < (kA + kB + kSf) / 16; i += kRateThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();  // the zeros are read by the tensor core
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  const uint32_t sf_col = tmem + 256;  // columns 256..: scale tiles

  if (threadIdx.x == 0) {
    uint32_t idesc;
    if constexpr (FMT == kFmtBF16) idesc = idesc_bf16(128, N);
    else if constexpr (FMT == kFmtNVFP4) idesc = idesc_nvf4(128, N);
    else idesc = idesc_mxf8(128, N, 0);
    if constexpr (FMT != kFmtBF16)
      for (int c = 0; c < 16; ++c) tc_copy_sf(sf_col + c * 4, desc_sf(smem_u32(sf + c * 512)));
    const uint32_t a0 = smem_u32(a), b0 = smem_u32(b);
    for (int it = 0; it < iters; ++it) {
      if constexpr (COPY_SF && FMT == kFmtNVFP4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          tc_copy_sf(sf_col + j * 8, desc_sf(smem_u32(sf + (4 + j) * 512)));
          tc_copy_sf(sf_col + j * 8 + 4, desc_sf(smem_u32(sf + j * 512)));
        }
      } else if constexpr (COPY_SF && FMT == kFmtMXFP8) {
        tc_copy_sf(sf_col, desc_sf(smem_u32(sf)));
        tc_copy_sf(sf_col + 4, desc_sf(smem_u32(sf + 512)));
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t da = desc_sw128(a0 + j * 32), db = desc_sw128(b0 + j * 32);
        const uint32_t acc = (it | j) != 0;
        if constexpr (FMT == kFmtBF16) mma_bf16(tmem, da, db, idesc, acc);
        else if constexpr (FMT == kFmtNVFP4)
          mma_nvf4(tmem, da, db, idesc, sf_col + j * 8, sf_col + 32 + j * 8, acc);
        else mma_mxf8(tmem, da, db, idesc, sf_col + 4, sf_col + 32, acc);
      }
    }
    tc_commit(done);
    if (!mbar_wait(done, 0, nullptr)) report_status(&g_rate_status, kStatusTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tmem, 512);
}

template <int FMT, int N, bool COPY_SF>
cudaError_t run_rate(int iters, int grid, cudaStream_t s, float* ms) {
  constexpr int smem = 1024 + 128 * 128 + N * 128 + 16 * 512 + 64;
  auto k = mma_rate_kernel<FMT, N, COPY_SF>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaEvent_t ev[2];
  if ((e = cudaEventCreate(&ev[0])) != cudaSuccess) return e;
  if ((e = cudaEventCreate(&ev[1])) != cudaSuccess) {
    cudaEventDestroy(ev[0]);
    return e;
  }
  k<<<grid, kRateThreads, smem, s>>>(iters / 8 + 1);  // warm-up
  cudaEventRecord(ev[0], s);
  k<<<grid, kRateThreads, smem, s>>>(iters);
  cudaEventRecord(ev[1], s);
  e = cudaEventSynchronize(ev[1]);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, ev[0], ev[1]);
  cudaEventDestroy(ev[0]);
  cudaEventDestroy(ev[1]);
  return e;
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_measure_mma_rate(int format, int n_cols, int copy_scales, int iters,
                                           double* tflops, void* stream) {
  if (!tflops || iters <= 0 || iters > (1 << 20) || (n_cols != 128 && n_cols != 256))
    return MOE_ERR_INVALID_ARG;
  if (format != MOE_FMT_BF16 && format != MOE_FMT_MXFP8 && format != MOE_FMT_NVFP4)
    return MOE_ERR_INVALID_ARG;
  if (copy_scales && (format == MOE_FMT_BF16 || n_cols != 128)) return MOE_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_NO_DEVICE;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_rate_status, &zero, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float ms = 0.0f;
  cudaError_t e;
  if (format == MOE_FMT_BF16)
    e = n_cols == 128 ? run_rate<kFmtBF16, 128, false>(iters, sms, s, &ms)
                      : run_rate<kFmtBF16, 256, false>(iters, sms, s, &ms);
  else if (format == MOE_FMT_MXFP8)
    e = n_cols == 256 ? run_rate<kFmtMXFP8, 256, false>(iters, sms, s, &ms)
        : copy_scales ? run_rate<kFmtMXFP8, 128, true>(iters, sms, s, &ms)
                      : run_rate<kFmtMXFP8, 128, false>(iters, sms, s, &ms);
  else
    e = n_cols == 256 ? run_rate<kFmtNVFP4, 256, false>(iters, sms, s, &ms)
        : copy_scales ? run_rate<kFmtNVFP4, 128, true>(iters, sms, s, &ms)
                      : run_rate<kFmtNVFP4, 128, false>(iters, sms, s, &ms);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  int st = 0;
  if (cudaMemcpyFromSymbol(&st, g_rate_status, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  if (st != 0) return MOE_ERR_DEVICE_TIMEOUT;
  const double k_elems = format == MOE_FMT_BF16 ? 16.0 : format == MOE_FMT_MXFP8 ? 32.0 : 64.0;
  const double flops = static_cast<double>(sms) * iters * 4.0 * 2.0 * 128.0 * n_cols * k_elems;
  *tflops = flops / (static_cast<double>(ms) * 1e-3) / 1e12;
  return MOE_OK;
}
