// pack.cu -- q1_0_pack / q1_0_unpack: 18-byte Q1_0 blocks <-> the packed
// device layout documented in common.cuh; q2_0_pack / q2_0_unpack: 34-byte
// Q2_0 blocks <-> the two-plane layout documented in q2.cuh.  Runs once per
// weight matrix.
#include "q2.cuh"

namespace q1 {

// Element of the 128-element block held by bit (8*i + pl) of word w: lane
// w + 4*(pl & 1) of sub-block pl >> 1, element i of the lane.
__device__ __forceinline__ int elem_of(int w, int pl, int i) {
  return 32 * (pl >> 1) + 4 * (w + 4 * (pl & 1)) + i;
}

// Per-call record of rejected input, in device memory the call allocates on
// its stream: the smallest (row * nb + block) index of a block whose fp16
// scale is Inf or NaN, and of a Q2_0 block holding the code 3 (all ones when
// there is none).
struct PackReject {
  unsigned long long scale;
  unsigned long long code;
};

__device__ __forceinline__ bool f16_nonfinite(uint16_t h) { return (h & 0x7c00u) == 0x7c00u; }

// One thread per (padded row, padded block).
__global__ void k_pack(const uint8_t* __restrict__ blocks, int64_t rows, int64_t nb, int64_t nbp,
                       int64_t rows_pad, uint32_t* __restrict__ bits, uint16_t* __restrict__ scales,
                       PackReject* __restrict__ reject) {
  int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows_pad * nbp) return;
  int64_t r = idx / nbp, b = idx % nbp;
  int64_t p = r / kPanel;
  int rr = int(r % kPanel);
  uint32_t word[4] = {0u, 0u, 0u, 0u};  // word w holds lanes w and w + 4
  uint16_t sc = 0;
  if (r < rows && b < nb) {
    const uint8_t* blk = blocks + (r * nb + b) * kBlockBytes;
    sc = uint16_t(blk[0] | (blk[1] << 8));
    if (f16_nonfinite(sc)) atomicMin(&reject->scale, (unsigned long long)(r * nb + b));
    uint8_t qs[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) qs[j] = blk[2 + j];
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
      for (int pl = 0; pl < 8; ++pl)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          int e = elem_of(w, pl, i);
          uint32_t bit = (qs[e >> 3] >> (e & 7)) & 1u;
          word[w] |= bit << (8 * i + pl);
        }
  }
#pragma unroll
  for (int w = 0; w < 4; ++w) bits[bits_word_index(p, b, rr, w, nbp)] = word[w];
  scales[scale_index(p, b, rr, nbp)] = sc;
}

// One thread per (row, block) of the real matrix.
__global__ void k_unpack(const uint32_t* __restrict__ bits, const uint16_t* __restrict__ scales,
                         int64_t rows, int64_t nb, int64_t nbp, uint8_t* __restrict__ blocks) {
  int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows * nb) return;
  int64_t r = idx / nb, b = idx % nb;
  int64_t p = r / kPanel;
  int rr = int(r % kPanel);
  uint8_t qs[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) qs[j] = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t word = bits[bits_word_index(p, b, rr, w, nbp)];
#pragma unroll
    for (int pl = 0; pl < 8; ++pl)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        int e = elem_of(w, pl, i);
        qs[e >> 3] |= uint8_t(((word >> (8 * i + pl)) & 1u) << (e & 7));
      }
  }
  uint16_t sc = scales[scale_index(p, b, rr, nbp)];
  uint8_t* blk = blocks + idx * kBlockBytes;
  blk[0] = uint8_t(sc & 0xff);
  blk[1] = uint8_t(sc >> 8);
#pragma unroll
  for (int j = 0; j < 16; ++j) blk[2 + j] = qs[j];
}

// Q2_0: one thread per (padded row, padded block); codes 0/1/2 become the N
// (weight -1) and P (+1) sign planes, each in the Q1_0 bit order.  A code 3
// (not a weight) is recorded in `reject` and packed as 0.
__global__ void k_pack_q2(const uint8_t* __restrict__ blocks, int64_t rows, int64_t nb, int64_t nbp,
                          int64_t rows_pad, uint32_t* __restrict__ bits, uint16_t* __restrict__ scales,
                          PackReject* __restrict__ reject) {
  int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows_pad * nbp) return;
  int64_t r = idx / nbp, b = idx % nbp;
  int64_t p = r / kPanel;
  int rr = int(r % kPanel);
  uint32_t pw[4] = {0u, 0u, 0u, 0u}, nw[4] = {0u, 0u, 0u, 0u};
  uint16_t sc = 0;
  if (r < rows && b < nb) {
    const uint8_t* blk = blocks + (r * nb + b) * 34;
    sc = uint16_t(blk[0] | (blk[1] << 8));
    if (f16_nonfinite(sc)) atomicMin(&reject->scale, (unsigned long long)(r * nb + b));
    uint8_t qs[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) qs[j] = blk[2 + j];
    bool bad = false;
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
      for (int pl = 0; pl < 8; ++pl)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int e = elem_of(w, pl, i);
          const uint32_t c = (qs[e >> 2] >> (2 * (e & 3))) & 3u;
          pw[w] |= uint32_t(c == 2u) << (8 * i + pl);
          nw[w] |= uint32_t(c == 0u) << (8 * i + pl);
          bad |= c == 3u;
        }
    if (bad) atomicMin(&reject->code, (unsigned long long)(r * nb + b));
  }
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    bits[q2_bits_word_index(p, b, rr, w, nbp, 0)] = pw[w];
    bits[q2_bits_word_index(p, b, rr, w, nbp, 1)] = nw[w];
  }
  scales[scale_index(p, b, rr, nbp)] = sc;
}

__global__ void k_unpack_q2(const uint32_t* __restrict__ bits, const uint16_t* __restrict__ scales,
                            int64_t rows, int64_t nb, int64_t nbp, uint8_t* __restrict__ blocks) {
  int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows * nb) return;
  int64_t r = idx / nb, b = idx % nb;
  int64_t p = r / kPanel;
  int rr = int(r % kPanel);
  uint8_t qs[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) qs[j] = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t P = bits[q2_bits_word_index(p, b, rr, w, nbp, 0)];
    const uint32_t N = bits[q2_bits_word_index(p, b, rr, w, nbp, 1)];
#pragma unroll
    for (int pl = 0; pl < 8; ++pl)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = elem_of(w, pl, i);
        const uint32_t pos = (P >> (8 * i + pl)) & 1u, neg = (N >> (8 * i + pl)) & 1u;
        const uint32_t c = pos ? 2u : (neg ? 0u : 1u);
        qs[e >> 2] |= uint8_t(c << (2 * (e & 3)));
      }
  }
  const uint16_t sc = scales[scale_index(p, b, rr, nbp)];
  uint8_t* blk = blocks + idx * 34;
  blk[0] = uint8_t(sc & 0xff);
  blk[1] = uint8_t(sc >> 8);
#pragma unroll
  for (int j = 0; j < 32; ++j) blk[2 + j] = qs[j];
}

static int check_pack_args(const char* who, const void* blocks, int64_t rows, int64_t n, const void* packed) {
  if (rows < 1 || rows > (int64_t(1) << 26) || n < 128 || n > (int64_t(1) << 24) || n % 128)
    return fail(Q1_ERR_ARG, "%s: bad shape rows=%lld n=%lld", who, (long long)rows, (long long)n);
  if (!blocks || !packed) return fail(Q1_ERR_ARG, "%s: null pointer", who);
  if (reinterpret_cast<uintptr_t>(blocks) % 2) return fail(Q1_ERR_ARG, "%s: blocks not 2-byte aligned", who);
  if (reinterpret_cast<uintptr_t>(packed) % 16) return fail(Q1_ERR_ARG, "%s: packed not 16-byte aligned", who);
  return Q1_OK;
}

// Runs one pack kernel with a fresh reject record on `s`, waits for it, and
// turns a recorded block into a Q1_ERR_ARG naming its row and block.  The
// record is this call's own (stream-ordered allocation), so calls on other
// threads or streams never see each other's findings.
template <class Launch>
static int pack_checked(const char* who, int64_t nb, cudaStream_t s, Launch&& launch) {
  PackReject* rec = nullptr;
  if (int e = cuda_status(cudaMallocAsync(reinterpret_cast<void**>(&rec), sizeof(PackReject), s), who)) return e;
  int rc = cuda_status(cudaMemsetAsync(rec, 0xff, sizeof(PackReject), s), who);
  if (rc == Q1_OK) rc = launch(rec);
  PackReject host = {~0ull, ~0ull};
  if (rc == Q1_OK) rc = cuda_status(cudaMemcpyAsync(&host, rec, sizeof host, cudaMemcpyDeviceToHost, s), who);
  const int rf = cuda_status(cudaFreeAsync(rec, s), who);
  // The products may read packed weights before the kernel that precedes them
  // on a stream has finished, so packing completes before the call returns;
  // the reject record needs the wait too.
  const int rs = cuda_status(cudaStreamSynchronize(s), who);
  if (rc != Q1_OK) return rc;
  if (rf != Q1_OK) return rf;
  if (rs != Q1_OK) return rs;
  if (host.scale != ~0ull)
    return fail(Q1_ERR_ARG, "%s: row %lld block %lld: the fp16 weight scale is not finite", who,
                (long long)(host.scale / nb), (long long)(host.scale % nb));
  if (host.code != ~0ull)
    return fail(Q1_ERR_ARG, "%s: row %lld block %lld holds the code 3, which is not a ternary weight", who,
                (long long)(host.code / nb), (long long)(host.code % nb));
  return Q1_OK;
}

}  // namespace q1

using namespace q1;

extern "C" int q1_0_pack(const uint8_t* blocks, int64_t rows, int64_t n, void* packed, void* stream) {
  if (int e = check_pack_args("q1_0_pack", blocks, rows, n, packed)) return e;
  Layout L = layout_of(rows, n);
  uint32_t* bits = static_cast<uint32_t*>(packed);
  uint16_t* scales = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(packed) + L.bits_bytes);
  int64_t total = L.rows_pad * L.nbp;
  int threads = 256;
  int64_t grid = (total + threads - 1) / threads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return pack_checked("q1_0_pack", L.nb, s, [&](PackReject* rec) {
    return launch_plain(k_pack, dim3(unsigned(grid)), dim3(threads), s, "q1_0_pack launch", blocks, rows, L.nb, L.nbp,
                        L.rows_pad, bits, scales, rec);
  });
}

extern "C" int q1_0_unpack(const void* packed, int64_t rows, int64_t n, uint8_t* blocks, void* stream) {
  if (int e = check_pack_args("q1_0_unpack", blocks, rows, n, packed)) return e;
  Layout L = layout_of(rows, n);
  const uint32_t* bits = static_cast<const uint32_t*>(packed);
  const uint16_t* scales =
      reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(packed) + L.bits_bytes);
  int64_t total = rows * L.nb;
  int threads = 256;
  int64_t grid = (total + threads - 1) / threads;
  return launch_plain(k_unpack, dim3(unsigned(grid)), dim3(threads), static_cast<cudaStream_t>(stream),
                      "q1_0_unpack launch", bits, scales, rows, L.nb, L.nbp, blocks);
}

extern "C" int q2_0_pack(const uint8_t* blocks, int64_t rows, int64_t n, void* packed, void* stream) {
  if (int e = check_pack_args("q2_0_pack", blocks, rows, n, packed)) return e;
  Layout L = layout_q2(rows, n);
  uint32_t* bits = static_cast<uint32_t*>(packed);
  uint16_t* scales = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(packed) + L.bits_bytes);
  int64_t total = L.rows_pad * L.nbp;
  int threads = 256;
  int64_t grid = (total + threads - 1) / threads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return pack_checked("q2_0_pack", L.nb, s, [&](PackReject* rec) {
    return launch_plain(k_pack_q2, dim3(unsigned(grid)), dim3(threads), s, "q2_0_pack launch", blocks, rows, L.nb,
                        L.nbp, L.rows_pad, bits, scales, rec);
  });
}

extern "C" int q2_0_unpack(const void* packed, int64_t rows, int64_t n, uint8_t* blocks, void* stream) {
  if (int e = check_pack_args("q2_0_unpack", blocks, rows, n, packed)) return e;
  Layout L = layout_q2(rows, n);
  const uint32_t* bits = static_cast<const uint32_t*>(packed);
  const uint16_t* scales =
      reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(packed) + L.bits_bytes);
  int64_t total = rows * L.nb;
  int threads = 256;
  int64_t grid = (total + threads - 1) / threads;
  return launch_plain(k_unpack_q2, dim3(unsigned(grid)), dim3(threads), static_cast<cudaStream_t>(stream),
                      "q2_0_unpack launch", bits, scales, rows, L.nb, L.nbp, blocks);
}
