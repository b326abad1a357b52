// common.cuh -- shared definitions of the CUDA path: packed weight layout,
// inline-PTX helpers, error reporting.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "q1gemv.h"

namespace q1 {

// ----------------------------------------------------------------- format --
constexpr int kBlock = 128;       // weights per Q1_0 block
constexpr int kBlockBytes = 18;   // fp16 scale + 16 sign bytes
constexpr int kSub = 32;          // activation values per q8_0 scale
constexpr int kPanel = 32;        // rows per panel
constexpr int kGroup = 8;         // panels per panel group (256 rows)
constexpr int kBlockPad = 4;      // blocks per row are padded to a multiple of 4 (a quad)

// Packed device layout (q1_0_pack writes it, the product kernels read it):
//
//   rows_pad = round_up(rows, 256), nbp = round_up(n/128, 4), nq = nbp/4,
//   panels = rows_pad/32, groups = rows_pad/256.
//
//   bits   : u32 words at byte 0.  For panel group gi, block quad qd (blocks
//            4qd..4qd+3), panel pi within the group (0..7), panel row r (0..31),
//            word w (0..3) and block bq within the quad, the word sits at
//              ((((gi*nq + qd)*8 + pi)*32 + r)*4 + w)*4 + bq
//            so one quad of one panel is 2 KB, a warp's 8 rows x 4 words
//            read 512 contiguous bytes, and the quad of 2, 4 or 8 aligned
//            consecutive panels is one contiguous 4, 8 or 16 KB chunk.
//   scales : fp16 block scales d0 after the bits (byte offset rows_pad*nbp*16),
//            half index (((gi*nq + qd)*8 + pi)*32 + r)*4 + bq: 256 B per panel
//            and quad, contiguous across the panels of a group in the same way.
//
// Within word w of (row, block): bit 8*i + pl (i = 0..3, plane pl = 0..7) is
// the sign bit of block element 32*(pl>>1) + 4*(w + 4*(pl&1)) + i, i.e. element
// i of lane w (even planes) or lane w + 4 (odd planes) of sub-block pl>>1.
// Masking a word with 0x01010101 << pl leaves that lane-and-sub-block's four
// sign bits as four bytes of value 0 or 2^pl.  Padded rows and blocks hold
// zero bits and zero scales.
struct Layout {
  int64_t rows, n, nb, nbp, panels, rows_pad;
  int64_t bits_bytes, scales_bytes, total_bytes;
};

inline Layout layout_of(int64_t rows, int64_t n) {
  Layout L;
  L.rows = rows;
  L.n = n;
  L.nb = n / kBlock;
  L.nbp = (L.nb + kBlockPad - 1) / kBlockPad * kBlockPad;
  L.rows_pad = (rows + kPanel * kGroup - 1) / (kPanel * kGroup) * (kPanel * kGroup);
  L.panels = L.rows_pad / kPanel;
  L.bits_bytes = L.rows_pad * L.nbp * 16;
  L.scales_bytes = L.rows_pad * L.nbp * 2;
  L.total_bytes = L.bits_bytes + L.scales_bytes;
  return L;
}

// Word index of (panel p, block b, panel row r, word w) and half index of
// the scale of (panel p, block b, row r); p counts panels from the start.
__host__ __device__ __forceinline__ int64_t bits_word_index(int64_t p, int64_t b, int r, int w, int64_t nbp) {
  return ((((p / kGroup) * (nbp / 4) + b / 4) * kGroup + p % kGroup) * kPanel + r) * 16 + w * 4 + (b % 4);
}
__host__ __device__ __forceinline__ int64_t scale_index(int64_t p, int64_t b, int r, int64_t nbp) {
  return ((((p / kGroup) * (nbp / 4) + b / 4) * kGroup + p % kGroup) * kPanel + r) * 4 + (b % 4);
}
// Byte offsets of the quad qd of panel p within the bits and scales regions.
__host__ __device__ __forceinline__ int64_t quad_bits_offset(int64_t p, int64_t qd, int64_t nbp) {
  return (((p / kGroup) * (nbp / 4) + qd) * kGroup + p % kGroup) * 2048;
}
__host__ __device__ __forceinline__ int64_t quad_scales_offset(int64_t p, int64_t qd, int64_t nbp) {
  return (((p / kGroup) * (nbp / 4) + qd) * kGroup + p % kGroup) * 256;
}

// Magic accumulator: the float whose bits are 0x4B400000 is 1.5 * 2^23 = C; for
// |t| < 2^22 the bits 0x4B400000 + t are the float C + t exactly.
constexpr uint32_t kMagicBits = 0x4B400000u;
constexpr float kMagic = 12582912.0f;

// ------------------------------------------------------------ PTX helpers --
__device__ __forceinline__ uint32_t dp4a_us(uint32_t a, uint32_t b, uint32_t c) {
  // c + sum_i a.u8[i] * b.s8[i]  (a unsigned bytes, b signed bytes)
  uint32_t d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Programmatic dependent launch: wait for the preceding kernel's memory, and
// allow the next kernel in the stream to begin launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------- error record --
// Sets the thread-local last-error text; returns `code`.
int fail(int code, const char* fmt, ...);
// Checks a CUDA runtime status after a launch; records and maps errors.
int cuda_status(cudaError_t e, const char* what);
// A plain launch (no attributes) whose status is that of this launch alone:
// unlike a <<<>>> launch checked with cudaGetLastError, an error an earlier
// call left behind is not taken for this launch's.
template <typename... KArgs, typename... Args>
int launch_plain(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s, const char* who, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  return cuda_status(cudaLaunchKernelEx(&cfg, kernel, args...), who);
}
// SM count of the current device (cached per device).
int num_sms();
// Argument checks of one q1_product (shape, pointers, 16-byte alignment).
int check_product(const char* who, int idx, const q1_product& pr);
// Device byte ranges a product launch pulls into L2 while it runs (the packed
// weights and the activation of the launch that follows): each p 16-byte
// aligned, bytes a multiple of 16; count 0 for none.
struct L2Range {
  const uint8_t* p;
  int64_t bytes;
};
struct L2Ranges {
  L2Range r[Q1_MAX_PREFETCH_RANGES];
  int count;
};
// The streaming matrix-vector kernel behind q1_0_gemv / q1_0_gemv_multi.
int launch_products_dp4a(const q1_product* prods, int count, cudaStream_t s, const char* who,
                         const L2Ranges& pf = L2Ranges{});
// Device status word of the product kernels (read and optionally cleared).
int status_word_dp4a(unsigned* v, int clear);
int status_word_prod(unsigned* v, int clear);
int status_word_tc(unsigned* v, int clear);
// The batched product on the tensor core (tcprod.cu): scratch bytes it needs
// for n and nvec, and the launch (a prologue kernel and the product kernel)
// with that scratch in device memory owned by the caller of launch_tc.
int64_t tc_scratch_bytes(int64_t n, int64_t nvec);
int launch_tc(const void* packed, int64_t rows, int64_t n, int64_t nvec, const int8_t* q, const uint16_t* d,
              float* out, uint8_t* scratch, cudaStream_t s, const char* who);

}  // namespace q1

namespace q1 {

// ------------------------------------------------ mbarrier / bulk copy ----
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait until the barrier's phase with parity `parity` has completed.  Bounded:
// gives up after about `limit_ns` nanoseconds and returns false (the clock is
// read only every 64 polls).
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done) : "r"(bar), "r"(parity) : "memory");
  return done != 0;
}

static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 63) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
  if (mbar_try(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, limit_ns);
}

// This CTA's share of an L2 prefetch of r, issued by the calling thread: the
// range is cut into `ctas` pieces on 16-byte boundaries and piece `cta` goes
// out as one bulk prefetch (one per 16 MB).  A hint: nothing waits for it.
__device__ __forceinline__ void l2_prefetch_share(const L2Range& r, int cta, int ctas) {
  if (r.p == nullptr || r.bytes < 16) return;
  const int64_t units = r.bytes >> 4;
  const int64_t u0 = units * cta / ctas, u1 = units * (cta + 1) / ctas;
  for (int64_t u = u0; u < u1; u += int64_t(1) << 20) {  // at most 16 MB an instruction
    const int64_t m = u1 - u < (int64_t(1) << 20) ? u1 - u : int64_t(1) << 20;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(r.p + (u << 4)), "r"(uint32_t(m << 4))
                 : "memory");
  }
}
__device__ __forceinline__ void l2_prefetch_share(const L2Ranges& rs, int cta, int ctas) {
  for (int i = 0; i < rs.count && i < Q1_MAX_PREFETCH_RANGES; ++i) l2_prefetch_share(rs.r[i], cta, ctas);
}

// 1-D bulk copy global -> shared, completing on `bar` (both addresses 16-byte
// aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Device status flags: a kernel whose bounded wait gives up ORs this into the
// library's device status word (read with q1_device_status) instead of hanging.
constexpr unsigned kStatusWaitTimeout = 1u;

}  // namespace q1
