// gemv.cu -- q1_0_gemm_small: the Q1_0 x q8_0 row product for up to 64
// activation vectors sharing one pass over the weights.
//
// Definition (bankML "docs/modules/gpu.md", "kernels.rs -- the Q1_0 kernels",
// first bullet) and the exactness argument are in table.cuh; out[v][r] is the
// matrix-vector product of row r and vector v.  A thread owns R rows (one per
// panel) and one lane pair, and keeps V vectors' chains; the activation
// constants of the V vectors sit in shared memory, chunk by chunk along n.
// The CTA's R panels arrive a quad of blocks at a time (R x 2.25 KB, two
// contiguous bulk copies thanks to the packed layout) in a ring of
// kProdStages shared-memory stages that one thread keeps filled, so the
// weight loads' latency is hidden without holding the next quad in registers.
#include <algorithm>
#include <atomic>
#include <cmath>

#include "table.cuh"

namespace q1 {

constexpr int kThreads = 128;  // 4 warps; thread (row in panel, lane pair)
constexpr int kProdStages = 3;                 // quads of weights in flight per CTA
static __device__ unsigned g_status_prod = 0u;  // bit 0: a bounded wait gave up

struct ProdArgs {
  const uint4* bits;     // packed sign words, 16-byte vectors
  const uint16_t* scales;  // packed fp16 block scales
  const int8_t* q;       // activation quants [nvec][n]
  const uint16_t* d1;    // activation scales [nvec][n/32]
  float* out;            // [nvec][rows]
  int64_t n;
  int rows, nb, nbp, panels, nvec;
  int vgroups;           // ceil(nvec / V)
  int kc;                // blocks per activation chunk held in shared memory
};

// R panels per CTA (each thread: R rows, one per panel, one lane pair) and
// V activation vectors per CTA.  1-D grid: bid = panel_group * vgroups + vgroup.
template <int R>
__host__ __device__ constexpr int prod_stage_bytes() { return R * (2048 + 256); }
template <int R, int V>
__host__ __device__ constexpr int prod_smem_bytes(int kc) {
  return kProdStages * prod_stage_bytes<R>() + 128 + V * table_bytes(kc);
}

template <int R, int V>
__global__ void __launch_bounds__(kThreads) k_q1_prod(ProdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int SB = prod_stage_bytes<R>();
  constexpr int S = kProdStages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * SB);
  unsigned char* tables = smem + S * SB + 128;
  // Table capacity in blocks, a compile-time stride between the vectors'
  // tables (the chunk a.kc never exceeds it).
  constexpr int KCM = (128 / V) / 8 * 8 > 8 ? (128 / V) / 8 * 8 : 8;
  constexpr int tb = table_bytes(KCM);
  const int lane = threadIdx.x & 31;
  const int w = lane & 3;                               // word w: lanes w and w+4
  const int prow = (threadIdx.x >> 5) * 8 + (lane >> 2);  // row within the panel

  const int vg = blockIdx.x % a.vgroups;
  const int pg = blockIdx.x / a.vgroups;
  const int p0 = pg * R;
  const int v0 = vg * V;
  const int nq = a.nbp / 4;  // quads of blocks along n (the panels are whole: R divides 8)
  const uint8_t* bits = reinterpret_cast<const uint8_t*>(a.bits);
  const uint8_t* scales = reinterpret_cast<const uint8_t*>(a.scales);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(smem_addr(&full[s]), 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Thread 0 keeps S quads of the CTA's R panels in flight (weights only:
  // they may be read before the preceding kernel has finished).
  auto issue = [&](int qd) {
    const int s = qd % S;
    const uint32_t bar = smem_addr(&full[s]);
    mbar_arrive_expect_tx(bar, uint32_t(SB));
    const uint32_t dst = smem_addr(smem + s * SB);
    bulk_g2s(dst, bits + quad_bits_offset(p0, qd, a.nbp), R * 2048, bar);
    bulk_g2s(dst + R * 2048, scales + quad_scales_offset(p0, qd, a.nbp), R * 256, bar);
  };
  if (threadIdx.x == 0)
    for (int qd = 0; qd < S && qd < nq; ++qd) issue(qd);

  pdl_wait();

  float accE[V][R], accO[V][R];  // lane w and lane w+4 chains
#pragma unroll
  for (int v = 0; v < V; ++v)
#pragma unroll
    for (int j = 0; j < R; ++j) accE[v][j] = accO[v][j] = 0.0f;

  bool ok = true;
  int waited = 0;  // quads whose stage this thread has seen complete
  for (int blk0 = 0; blk0 < a.nbp && ok; blk0 += a.kc) {
    const int kcb = min(a.kc, a.nbp - blk0);
    __syncthreads();
#pragma unroll
    for (int v = 0; v < V; ++v) {
      unsigned char* t = tables + v * tb;
      const int vv = min(v0 + v, a.nvec - 1);
      build_table_q<4>(a.q + int64_t(vv) * a.n, a.d1 + int64_t(vv) * (a.n / kSub), a.nb, blk0, kcb, t,
                       threadIdx.x, kThreads, KCM);
    }
    __syncthreads();

    for (int b = blk0; b < blk0 + kcb; b += 4) {
      const int qd = b / 4, s = qd % S;
      const bool got = mbar_wait(smem_addr(&full[s]), uint32_t(qd / S) & 1u);
      const unsigned char* st = smem + s * SB;
      uint4 wv[R];
      uint2 sc[R];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        wv[j] = got ? reinterpret_cast<const uint4*>(st + j * 2048)[prow * 4 + w] : make_uint4(0u, 0u, 0u, 0u);
        sc[j] = got ? reinterpret_cast<const uint2*>(st + R * 2048 + j * 256)[prow] : make_uint2(0u, 0u);
      }
      // Every thread holds its words: the stage may be refilled.  A wait that
      // gave up anywhere ends the loop for the whole CTA at the same point.
      if (__syncthreads_or(!got)) {
        ok = false;
        break;
      }
      waited = qd + 1;
      if (threadIdx.x == 0 && qd + S < nq) issue(qd + S);
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const unsigned char* t = tables + v * tb;
        quad_all<R>(wv, sc, reinterpret_cast<const uint4*>(t) + (b - blk0) * 16,
                    reinterpret_cast<const float4*>(t + table_dk_offset(KCM)) + (b - blk0) * 4, w, accE[v],
                    accO[v]);
      }
    }
  }
  if (!ok) {
    // Give the copies still in flight (all issued by thread 0) a bounded
    // chance to land before the CTA's shared memory goes away.
    atomicOr(&g_status_prod, kStatusWaitTimeout);
    if (threadIdx.x == 0)
      for (int qd = waited; qd < nq && qd < waited + S; ++qd)
        mbar_wait(smem_addr(&full[qd % S]), uint32_t(qd / S) & 1u, 100000000ull);
    return;
  }

  pdl_launch_dependents();
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int64_t row = int64_t(p0 + j) * kPanel + prow;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const float r = row_sum(accE[v][j], accO[v][j]);
      if (w == 0 && row < a.rows && v0 + v < a.nvec) a.out[int64_t(v0 + v) * a.rows + row] = r;
    }
  }
}

int status_word_prod(unsigned* v, int clear) {
  if (int e = cuda_status(cudaMemcpyFromSymbol(v, g_status_prod, sizeof *v), "q1_device_status")) return e;
  if (clear && *v) {
    const unsigned zero = 0;
    return cuda_status(cudaMemcpyToSymbol(g_status_prod, &zero, sizeof zero), "q1_device_status");
  }
  return Q1_OK;
}

template <int R, int V>
static int launch(const ProdArgs& a0, int64_t panels, cudaStream_t s, const char* who) {
  ProdArgs a = a0;
  a.vgroups = (a.nvec + V - 1) / V;
  a.kc = std::min<int>(a.nbp, std::max(8, (128 / V) / 8 * 8));
  const int64_t pgroups = (panels + R - 1) / R;
  const int64_t grid = pgroups * a.vgroups;
  if (grid > 0x7fffffff) return fail(Q1_ERR_ARG, "%s: matrix too large for one launch", who);
  const int smem = prod_smem_bytes<R, V>(std::max(8, (128 / V) / 8 * 8));
  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!attr_done[dev]) {
    if (int e = cuda_status(cudaFuncSetAttribute(k_q1_prod<R, V>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 prod_smem_bytes<R, V>(128)), "cudaFuncSetAttribute"))
      return e;
    attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, k_q1_prod<R, V>, a), who);
}

static int check_prod_args(const char* who, const void* packed, int64_t rows, int64_t n, int64_t nvec,
                           const int8_t* q, const uint16_t* d, const float* out) {
  if (rows < 1 || rows > (int64_t(1) << 26) || n < 128 || n > (int64_t(1) << 24) || n % 128)
    return fail(Q1_ERR_ARG, "%s: bad shape rows=%lld n=%lld", who, (long long)rows, (long long)n);
  if (nvec < 1 || nvec > 64) return fail(Q1_ERR_ARG, "%s: nvec=%lld outside 1..64", who, (long long)nvec);
  if (!packed || !q || !d || !out) return fail(Q1_ERR_ARG, "%s: null pointer", who);
  if (reinterpret_cast<uintptr_t>(packed) % 16 || reinterpret_cast<uintptr_t>(q) % 16 ||
      reinterpret_cast<uintptr_t>(d) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
    return fail(Q1_ERR_ARG, "%s: buffers must be 16-byte aligned", who);
  return Q1_OK;
}

static ProdArgs make_args(const void* packed, int64_t rows, int64_t n, int64_t nvec, const int8_t* q,
                          const uint16_t* d, float* out) {
  Layout L = layout_of(rows, n);
  ProdArgs a = {};
  a.bits = static_cast<const uint4*>(packed);
  a.scales = reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(packed) + L.bits_bytes);
  a.q = q;
  a.d1 = d;
  a.out = out;
  a.n = n;
  a.rows = int(rows);
  a.nb = int(L.nb);
  a.nbp = int(L.nbp);
  a.panels = int(L.panels);
  a.nvec = int(nvec);
  return a;
}

}  // namespace q1

using namespace q1;

// The stream-ordered pool the batched product takes its per-call scratch
// from, one per device.  Freed scratch stays in the pool for the next call
// (release threshold: unlimited) instead of going back to the driver at every
// synchronization, which made each call pay a fresh allocation; the pool
// holds at most the largest scratch of concurrently running calls.
static int scratch_pool(cudaMemPool_t* out) {
  static cudaMemPool_t pools[64] = {};
  int dev = 0;
  if (int e = cuda_status(cudaGetDevice(&dev), "q1_0_gemm_small")) return e;
  if (dev < 0 || dev >= 64) return fail(Q1_ERR_ARG, "q1_0_gemm_small: device %d outside 0..63", dev);
  if (!pools[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t p = nullptr;
    if (int e = cuda_status(cudaMemPoolCreate(&p, &props), "q1_0_gemm_small: cudaMemPoolCreate")) return e;
    uint64_t keep = ~uint64_t(0);
    if (int e = cuda_status(cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep),
                            "q1_0_gemm_small: cudaMemPoolSetAttribute"))
      return e;
    pools[dev] = p;
  }
  *out = pools[dev];
  return Q1_OK;
}

// Which kernel is faster for a product, from a cost model of both measured on
// a GB300 (cold L2, one launch between events; 14336x4096 to 128256x4096,
// 8 to 64 vectors): the tensor-core kernel keeps one 128-row x 16-vector
// unit per SM in flight at about 0.51 us per block of 128 weights, plus
// about 12 us of prologue and ramp; the dp4a kernel streams about 2.2e13
// weight-vector products per second plus about 5 us.
static bool tc_faster(int64_t rows, int64_t n, int64_t nvec) {
  const double sms = double(num_sms());
  const double units = double((rows + 127) / 128) * double((nvec + 15) / 16);
  const double waves = std::ceil(units / sms);
  const double t_tc = waves * double(n / kBlock) * 0.51 + 12.0;
  const double t_dp4a = double(rows) * double(n) * double(nvec) / 2.2e7 + 5.0;
  return t_tc < t_dp4a;
}

// Vector counts from which the tensor-core kernel (tcprod.cu) takes the
// product, and the largest scratch it may ask for (records of 8 KB per block
// and group of 16 vectors: up to 64 MB at n = 2^20 and 64 vectors).
constexpr int64_t kTcMinVectors = 8;
constexpr int64_t kTcMaxScratch = int64_t(64) << 20;

// Kernel choice of q1_0_gemm_small (q1_gemm_small_kernel): 0 automatic, 1 dp4a,
// 2 tensor core.
static std::atomic<int> g_kernel_choice{0};

extern "C" int q1_gemm_small_kernel(int choice) {
  if (choice < 0 || choice > 2) return fail(Q1_ERR_ARG, "q1_gemm_small_kernel: choice %d outside 0..2", choice);
  return g_kernel_choice.exchange(choice);
}

extern "C" int q1_0_gemm_small(const void* packed, int64_t rows, int64_t n, int64_t nvec, const int8_t* q,
                               const uint16_t* d, float* out, void* stream) {
  if (int e = check_prod_args("q1_0_gemm_small", packed, rows, n, nvec, q, d, out)) return e;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t scratch_bytes = tc_scratch_bytes(n, nvec);
  const int choice = g_kernel_choice.load();
  if (choice == 2 && scratch_bytes > kTcMaxScratch)
    return fail(Q1_ERR_ARG, "q1_0_gemm_small: the tensor-core kernel would need %lld bytes of scratch (limit %lld)",
                (long long)scratch_bytes, (long long)kTcMaxScratch);
  const bool tc = choice == 2 || (choice == 0 && nvec >= kTcMinVectors && scratch_bytes <= kTcMaxScratch &&
                                  tc_faster(rows, n, nvec));
  if (tc) {
    // The scratch lives for this call only (stream-ordered allocation from
    // the library's pool), so calls on different streams never share it.
    uint8_t* scratch = nullptr;
    cudaMemPool_t pool = nullptr;
    if (int e = scratch_pool(&pool)) return e;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&scratch), size_t(scratch_bytes), pool, s) != cudaSuccess) {
      (void)cudaGetLastError();
      return fail(Q1_ERR_NOMEM, "q1_0_gemm_small: could not allocate %lld bytes of scratch on the stream",
                  (long long)scratch_bytes);
    }
    const int rc = launch_tc(packed, rows, n, nvec, q, d, out, scratch, s, "q1_0_gemm_small launch");
    const int rf = cuda_status(cudaFreeAsync(scratch, s), "q1_0_gemm_small");
    return rc != Q1_OK ? rc : rf;
  }
  ProdArgs a = make_args(packed, rows, n, nvec, q, d, out);
  const int64_t panels = a.panels;
  // Four rows per thread amortize each activation-table load over four rows
  // (one row per thread leaves the loop bound by shared-memory loads).  Four
  // vectors per CTA, or two when that leaves fewer than two CTAs per SM.
  if (nvec == 1) return launch<1, 1>(a, panels, s, "q1_0_gemm_small launch");
  const int64_t pgroups = (panels + 3) / 4;
  if (nvec <= 2 || pgroups * ((nvec + 3) / 4) < 2 * int64_t(num_sms()))
    return launch<4, 2>(a, panels, s, "q1_0_gemm_small launch");
  return launch<4, 4>(a, panels, s, "q1_0_gemm_small launch");
}
