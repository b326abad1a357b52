// quant.cu -- q8_quantize_act: q8_0 activation quantization, eight lanes per
// 32-value block.
#include "common.cuh"

namespace q1 {

// 256 threads = 8 warps; a warp takes four consecutive 32-value blocks, eight
// lanes a block, each lane one 16-byte load of four values (so a warp reads
// 512 contiguous bytes: full-width requests, which matters most when x is
// pinned host memory read over the host link).
constexpr int kQuantBlocksPerCta = 32;
__global__ void __launch_bounds__(256) k_quantize(const float* __restrict__ x, int64_t nblocks,
                                                  int8_t* __restrict__ q, uint16_t* __restrict__ d) {
  pdl_launch_dependents();
  pdl_wait();  // x may be written by the preceding kernel
  const int lane = threadIdx.x & 31;
  const int64_t blk0 = int64_t(blockIdx.x) * kQuantBlocksPerCta + (threadIdx.x >> 5) * 4;
  if (blk0 >= nblocks) return;  // whole warp
  const int64_t blk = blk0 + (lane >> 3);
  const bool live = blk < nblocks;
  const int64_t e = blk * kSub + (lane & 7) * 4;
  float4 v = live ? *reinterpret_cast<const float4*>(x + e) : make_float4(0.f, 0.f, 0.f, 0.f);
  float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (!live) return;
  float dd = __fdiv_rn(amax, 127.0f);
  float id = (dd != 0.0f) ? __fdiv_rn(1.0f, dd) : 0.0f;
  auto code = [&](float t) { return uint32_t(uint8_t(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(t, id)))))); };
  *reinterpret_cast<uint32_t*>(q + e) = code(v.x) | code(v.y) << 8 | code(v.z) << 16 | code(v.w) << 24;
  if ((lane & 7) == 0) d[blk] = __half_as_ushort(__float2half_rn(dd));
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
  cfg.gridDim = dim3(unsigned((nblocks + kQuantBlocksPerCta - 1) / kQuantBlocksPerCta));
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
