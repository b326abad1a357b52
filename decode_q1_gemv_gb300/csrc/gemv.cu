// gemv.cu -- q1_0_gemm_small: the Q1_0 x q8_0 row product for up to 64
// activation vectors sharing one pass over the weights.
//
// Definition (bankML "docs/modules/gpu.md", "kernels.rs -- the Q1_0 kernels",
// first bullet) and the exactness argument are in table.cuh; out[v][r] is the
// matrix-vector product of row r and vector v.  A thread owns R rows (one per
// panel) and one lane pair, and keeps V vectors' chains; the activation
// constants of the V vectors sit in shared memory, chunk by chunk along n.
#include <algorithm>

#include "table.cuh"

namespace q1 {

constexpr int kThreads = 128;  // 4 warps; thread (row in panel, lane pair)

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
template <int R, int V>
__global__ void __launch_bounds__(kThreads) k_q1_prod(ProdArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tb = table_bytes(a.kc);
  const int lane = threadIdx.x & 31;
  const int w = lane & 3;                               // word w: lanes w and w+4
  const int prow = (threadIdx.x >> 5) * 8 + (lane >> 2);  // row within the panel

  const int vg = blockIdx.x % a.vgroups;
  const int pg = blockIdx.x / a.vgroups;
  const int p0 = pg * R;
  const int v0 = vg * V;

  pdl_wait();

  float accE[V][R], accO[V][R];  // lane w and lane w+4 chains
#pragma unroll
  for (int v = 0; v < V; ++v)
#pragma unroll
    for (int j = 0; j < R; ++j) accE[v][j] = accO[v][j] = 0.0f;

  for (int blk0 = 0; blk0 < a.nbp; blk0 += a.kc) {
    const int kcb = min(a.kc, a.nbp - blk0);
    __syncthreads();
#pragma unroll
    for (int v = 0; v < V; ++v) {
      unsigned char* t = smem + v * tb;
      const int vv = min(v0 + v, a.nvec - 1);
      build_table_q<4>(a.q + int64_t(vv) * a.n, a.d1 + int64_t(vv) * (a.n / kSub), a.nb, blk0, kcb, t,
                    threadIdx.x, kThreads, a.kc);
    }
    __syncthreads();

    for (int b = blk0; b < blk0 + kcb; b += 4) {
      uint4 wv[R];
      uint2 sc[R];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int64_t p = p0 + j;
        if (p < a.panels) {
          wv[j] = ldg_stream(a.bits + bits_word_index(p, b, prow, w, a.nbp) / 4);
          sc[j] = *reinterpret_cast<const uint2*>(a.scales + scale_index(p, b, prow, a.nbp));
        } else {
          wv[j] = make_uint4(0u, 0u, 0u, 0u);
          sc[j] = make_uint2(0u, 0u);
        }
      }
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const unsigned char* t = smem + v * tb;
        quad_all<R>(wv, sc, reinterpret_cast<const uint4*>(t) + (b - blk0) * 16,
                    reinterpret_cast<const float4*>(t + table_dk_offset(a.kc)) + (b - blk0) * 4, w, accE[v],
                    accO[v]);
      }
    }
  }

  pdl_launch_dependents();
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int64_t row = int64_t(p0 + j) * kPanel + prow;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const float r = row_sum(accE[v][j], accO[v][j]);
      if (w == 0 && p0 + j < a.panels && row < a.rows && v0 + v < a.nvec)
        a.out[int64_t(v0 + v) * a.rows + row] = r;
    }
  }
}

template <int R, int V>
static int launch(const ProdArgs& a0, int64_t panels, cudaStream_t s, const char* who) {
  ProdArgs a = a0;
  a.vgroups = (a.nvec + V - 1) / V;
  a.kc = std::min<int>(a.nbp, std::max(8, (128 / V) / 8 * 8));
  const int64_t pgroups = (panels + R - 1) / R;
  const int64_t grid = pgroups * a.vgroups;
  if (grid > 0x7fffffff) return fail(Q1_ERR_ARG, "%s: matrix too large for one launch", who);
  const int smem = table_bytes(a.kc) * V;
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

extern "C" int q1_0_gemm_small(const void* packed, int64_t rows, int64_t n, int64_t nvec, const int8_t* q,
                               const uint16_t* d, float* out, void* stream) {
  if (int e = check_prod_args("q1_0_gemm_small", packed, rows, n, nvec, q, d, out)) return e;
  ProdArgs a = make_args(packed, rows, n, nvec, q, d, out);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
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
