// quant.cu -- q8_quantize_act: q8_0 activation quantization, one warp per
// 32-value block.
#include "common.cuh"

namespace q1 {

// 256 threads = 8 warps = 8 blocks of 32 values per CTA.
__global__ void __launch_bounds__(256) k_quantize(const float* __restrict__ x, int64_t nblocks,
                                                  int8_t* __restrict__ q, uint16_t* __restrict__ d) {
  pdl_launch_dependents();
  pdl_wait();  // x may be written by the preceding kernel
  int64_t blk = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  if (blk >= nblocks) return;
  float v = x[blk * kSub + lane];
  float amax = fabsf(v);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  float dd = __fdiv_rn(amax, 127.0f);
  float id = (dd != 0.0f) ? __fdiv_rn(1.0f, dd) : 0.0f;
  float t = __fmul_rn(v, id);
  q[blk * kSub + lane] = static_cast<int8_t>(static_cast<int>(roundf(t)));
  if (lane == 0) d[blk] = __half_as_ushort(__float2half_rn(dd));
}

}  // namespace q1

using namespace q1;

extern "C" int q8_quantize_act(const float* x, int64_t nvec, int64_t n, int8_t* q, uint16_t* d, void* stream) {
  if (nvec < 1 || nvec > 65535 || n < 32 || n > (int64_t(1) << 24) || n % 32)
    return fail(Q1_ERR_ARG, "q8_quantize_act: bad shape nvec=%lld n=%lld", (long long)nvec, (long long)n);
  if (!x || !q || !d) return fail(Q1_ERR_ARG, "q8_quantize_act: null pointer");
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(q) % 16 ||
      reinterpret_cast<uintptr_t>(d) % 16)
    return fail(Q1_ERR_ARG, "q8_quantize_act: buffers must be 16-byte aligned");
  int64_t nblocks = nvec * (n / kSub);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((nblocks + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, k_quantize, x, nblocks, q, d), "q8_quantize_act launch");
}
