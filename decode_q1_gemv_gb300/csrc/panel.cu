// panel.cu -- the matrix-vector product for one product of few rows: one CTA
// per 32-row panel, the panel's block quads shared out among its warps, which
// work on them at the same time.
//
// Row product (bankML "docs/modules/gpu.md", "kernels.rs -- the Q1_0
// kernels", first and second bullets): per lane, ab_b = d1*s summed over the
// four sub-blocks of block b, then acc = fma(d0_b, ab_b, acc) over the blocks
// in increasing order, then the fixed horizontal sum of the eight lanes.  Only
// the outer chain is sequential; ab_b depends on block b alone.
//
// The streaming kernel gives a tile of rows to one CTA, which walks all of n
// in sequence.  A product of a few thousand rows has fewer tiles than the GPU
// has SMs, and the few warps of each busy CTA mostly wait on their own
// dependences.  Here warp k of a panel's CTA takes a contiguous range of the
// quads: it loads their sign words and scales straight from global memory
// (issued before griddepcontrol.wait, as weights do not depend on the
// preceding kernel), builds the activation table entries of its own blocks
// (no CTA-wide barrier), forms ab_b for its blocks with the streaming kernel's
// quad step at four rows a thread (rows lane/4 + 8j, word lane%4), and leaves
// ab_b and d0_b in shared memory.  After one barrier the first four warps run
// the outer chain over all blocks in order and the horizontal sum: the same
// operations in the same order as the streaming kernel, so the same bits.
//
// Shared memory per CTA: the activation table of the whole row, ab as
// [block][row][word] float pairs (lanes w, w + 4) and d0 as [block][row]:
// 1472 bytes per block, so n up to 156 * 128 = 19968.  There are no waits on
// other CTAs or on asynchronous copies.
#include "formats.cuh"

namespace q1 {

namespace {

constexpr int kPanelBytesPerBlock = 4 * (4 * 16 + 16) + 128 * 8 + 32 * 4;  // table + ab + d0
constexpr int kPanelMaxNbp = 156;
constexpr int kPanelSmemPerSm = 233472;  // shared memory of an SM
constexpr int kPanelSmemPerCta = 1024;   // reserved by the system per resident CTA

constexpr int kPanelMaxProducts = 8;
constexpr int kPanelMaxPpc = 8;          // panels a CTA takes at most
constexpr int kPanelSmemMax = kPanelSmemPerSm - kPanelSmemPerCta;  // a CTA's dynamic shared memory at most

struct PanelProd {
  const uint8_t* packed;
  const float* x;        // f32 activation, or null
  const int8_t* q;       // q8_0 quants (when x is null)
  const uint16_t* d;     // q8_0 scales (when x is null)
  float* out;
  int64_t bits_bytes;
  int rows, nb, nbp;
  int panels;            // panels of the product (rows padded to panel groups)
  int panel_begin;       // first CTA of this product
};
struct PanelArgs {
  PanelProd p[kPanelMaxProducts];
  int count;
  int ppc;      // consecutive panels of a product per CTA (1: each warp builds its own table entries)
  L2Ranges pf;  // pulled into L2 while this launch runs (the next launch's inputs)
};

// Shared memory: one table for the row, and ab + d0 for each of the CTA's panels.
__host__ __device__ constexpr int panel_smem_bytes(int nbp, int ppc = 1) {
  return nbp * 4 * (4 * 16 + 16) + ppc * nbp * (128 * 8 + 32 * 4);
}

// fp16 scale w (0..3) of a quad held as 4 halves in a uint2.
__device__ __forceinline__ float quad_scale_at(const uint2& v, int w) {
  const uint32_t h = (w < 2) ? v.x : v.y;
  return __half2float(__ushort_as_half(uint16_t((w & 1) ? (h >> 16) : (h & 0xffffu))));
}

// Block BQ of a quad for four rows and word w: ab for lanes w (abE) and
// w + 4 (abO) of each row, stored to the CTA's ab array at [block][row][w].
template <class F, int BQ>
__device__ __forceinline__ void block_ab(const uint4 (&wv)[4], const uint4 (&nv)[4], const uint4* QCq,
                                         const float4* DKq, int w, int r0, float2* abq) {
  float abE[4], abO[4];
  if constexpr (F::kTwoPlanes) {
    q2_quad_subblock<4, BQ, 0>(wv, nv, QCq, DKq, w, abE, abO);
    q2_quad_subblock<4, BQ, 1>(wv, nv, QCq, DKq, w, abE, abO);
    q2_quad_subblock<4, BQ, 2>(wv, nv, QCq, DKq, w, abE, abO);
    q2_quad_subblock<4, BQ, 3>(wv, nv, QCq, DKq, w, abE, abO);
  } else {
    quad_subblock<4, BQ, 0>(wv, QCq, DKq, w, abE, abO);
    quad_subblock<4, BQ, 1>(wv, QCq, DKq, w, abE, abO);
    quad_subblock<4, BQ, 2>(wv, QCq, DKq, w, abE, abO);
    quad_subblock<4, BQ, 3>(wv, QCq, DKq, w, abE, abO);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) abq[(BQ * 32 + r0 + 8 * j) * 4 + w] = make_float2(abE[j], abO[j]);
}

// A unit of UB blocks (a quad, UB = 4, or half a quad, UB = 2) for rows
// r0 + 8j (j < 4) and word w: ab of its blocks, and the scale of block w of
// each row to the d0 array at [block][row] (threads w < UB).  wv/nv hold the
// unit's words in their first UB components, sc its scales in its first UB
// halves.
template <class F, int UB>
__device__ __forceinline__ void unit_ab(const uint4 (&wv)[4], const uint4 (&nv)[4], const uint2 (&sc)[4],
                                        const uint4* QCq, const float4* DKq, int w, int r0, float2* abq,
                                        float* d0q) {
  block_ab<F, 0>(wv, nv, QCq, DKq, w, r0, abq);
  block_ab<F, 1>(wv, nv, QCq, DKq, w, r0, abq);
  if constexpr (UB == 4) {
    block_ab<F, 2>(wv, nv, QCq, DKq, w, r0, abq);
    block_ab<F, 3>(wv, nv, QCq, DKq, w, r0, abq);
  }
  if (w < UB) {
#pragma unroll
    for (int j = 0; j < 4; ++j) d0q[w * 32 + r0 + 8 * j] = quad_scale_at(sc[j], w);
  }
}

// Register budget of a thread (the prefetched words of PF units dominate) and
// the CTAs of W warps an SM holds at that budget (at least one).  The kernel's
// launch bounds ask for that many CTAs an SM, which holds the compiler to the
// budget; where that is one CTA (16 warps) it may use up to 128 registers.
template <class F>
__host__ __device__ constexpr int panel_regs() { return F::kTwoPlanes ? 128 : 80; }
template <class F>
__host__ __device__ constexpr int panel_ctas_by_regs(int W) {
  return 65536 / (panel_regs<F>() * 32 * W) > 0 ? 65536 / (panel_regs<F>() * 32 * W) : 1;
}

// W warps; the panel's blocks form units of UB blocks (UB = 4: quads; UB = 2:
// half quads, for rows of few quads, so that more warps get work).  Warp k
// takes the contiguous units [k m, k m + m) (m = ceil(units / W)), four rows a
// thread, keeps the words of PF units in flight, and builds the activation
// table entries of its own blocks.  A CTA may take a.ppc consecutive panels
// of one product (the units of all of them, panel by panel): it then builds
// the whole table once, with all its threads, before the quad steps.
template <class F, int W, int PF, int UB, bool MP>
__global__ void __launch_bounds__(32 * W, panel_ctas_by_regs<F>(W)) k_q1_panel(const __grid_constant__ PanelArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  int j = 0;  // this CTA's product: panels are numbered across the products in list order
  while (j + 1 < a.count && int(blockIdx.x) >= a.p[j + 1].panel_begin) ++j;
  const PanelProd& pr = a.p[j];
  const int ppc = MP ? a.ppc : 1;  // the one-panel instance keeps the unit arithmetic compile-time
  const int nbp = pr.nbp, nu = nbp / UB;
  unsigned char* table = smem;
  float2* ab = reinterpret_cast<float2*>(smem + table_bytes(nbp));  // [panel][block][row][word]
  float* d0s = reinterpret_cast<float*>(ab + ppc * nbp * 128);      // [panel][block][row]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = lane >> 2, w = lane & 3;  // rows r0 + 8j of the panel, word w
  const int64_t p0 = int64_t(int(blockIdx.x) - pr.panel_begin) * ppc;  // first panel of this CTA
  const int np = !MP ? 1 : pr.panels - int(p0) < ppc ? pr.panels - int(p0) : ppc;  // its panels
  const int nunits = np * nu;
  const uint8_t* bits = pr.packed;
  const uint8_t* scales = pr.packed + pr.bits_bytes;
  const int m = (nunits + W - 1) / W;
  const int u0 = warp * m < nunits ? warp * m : nunits;
  const int mine = u0 + m < nunits ? m : nunits - u0;  // units [u0, u0 + mine) of this warp

  // Sign words are loaded ahead; the block scales, needed only when a unit's
  // products are stored, are loaded as its step starts.  Unit u is of panel
  // u / nu; within it, quad uu UB / 4, blocks (uu UB) % 4 .. + UB - 1
  // (uu = u % nu).
  uint4 wv[PF][4], nv[PF][4];
  auto load = [&](int i0) {
#pragma unroll
    for (int v = 0; v < PF; ++v) {
      if (i0 + v < mine) {
        const int u = u0 + i0 + v, pi = MP ? u / nu : 0, uu = u - pi * nu, qd = uu * UB / 4, h = (uu * UB) % 4 / 2;
        const uint8_t* rec = bits + F::quad_bits_offset(p0 + pi, qd, nbp);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int word = (r0 + 8 * j) * 4 + w;
          if constexpr (UB == 4) {
            wv[v][j] = __ldg(reinterpret_cast<const uint4*>(rec) + word);
            if constexpr (F::kTwoPlanes) nv[v][j] = __ldg(reinterpret_cast<const uint4*>(rec + 2048) + word);
          } else {
            const uint2 x2 = __ldg(reinterpret_cast<const uint2*>(rec) + word * 2 + h);
            wv[v][j] = make_uint4(x2.x, x2.y, 0u, 0u);
            if constexpr (F::kTwoPlanes) {
              const uint2 n2 = __ldg(reinterpret_cast<const uint2*>(rec + 2048) + word * 2 + h);
              nv[v][j] = make_uint4(n2.x, n2.y, 0u, 0u);
            }
          }
        }
      }
    }
  };
  load(0);
  // The next launch's inputs (q1_0_gemv_multi_prefetch), one bulk prefetch a
  // range from one thread: spread over a warp's lanes they held that warp back.
  if (tid == 32 * W - 32) l2_prefetch_share(a.pf, int(blockIdx.x), int(gridDim.x));

  pdl_wait();  // the activation may be written by the preceding kernel
  if (!MP) {
    if (mine > 0) {  // this warp's own table entries: blocks UB u0 .. UB (u0 + mine) - 1
      // Inlined, so that the sign-word loads above stay in flight meanwhile.
      if (pr.x) table_x_body<2, typename F::Consts>(pr.x, pr.nb, UB * u0, UB * mine, table, lane, 32, nbp, UB * u0);
      else table_q_body<4, typename F::Consts>(pr.q, pr.d, pr.nb, UB * u0, UB * mine, table, lane, 32, nbp, UB * u0);
    }
    __syncwarp();
  } else {  // the whole table, once for the CTA's panels, by all its threads
    if (pr.x) table_x_body<2, typename F::Consts>(pr.x, pr.nb, 0, nbp, table, tid, 32 * W, nbp, 0);
    else table_q_body<4, typename F::Consts>(pr.q, pr.d, pr.nb, 0, nbp, table, tid, 32 * W, nbp, 0);
    __syncthreads();
  }

  const uint4* QC = reinterpret_cast<const uint4*>(table);
  const float4* DK = reinterpret_cast<const float4*>(table + table_dk_offset(nbp));
  for (int i0 = 0; i0 < mine; i0 += PF) {
    if (i0 > 0) load(i0);
#pragma unroll
    for (int v = 0; v < PF; ++v) {
      if (i0 + v < mine) {
        const int u = u0 + i0 + v, pi = MP ? u / nu : 0, uu = u - pi * nu, qd = uu * UB / 4, h = (uu * UB) % 4 / 2;
        const int b0 = uu * UB;
        const uint2* srec = reinterpret_cast<const uint2*>(scales + quad_scales_offset(p0 + pi, qd, nbp));
        uint2 sc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if constexpr (UB == 4) sc[j] = __ldg(srec + r0 + 8 * j);
          else sc[j] = make_uint2(__ldg(reinterpret_cast<const uint32_t*>(srec + r0 + 8 * j) + h), 0u);
        }
        unit_ab<F, UB>(wv[v], nv[v], sc, QC + b0 * 16, DK + b0 * 4, w, r0, ab + (pi * nbp + b0) * 128,
                       d0s + (pi * nbp + b0) * 32);
      }
    }
  }
  pdl_launch_dependents();
  __syncthreads();

  // Outer chain over all blocks in order: (panel, row, word) per thread,
  // lanes w and w + 4 (idx % 4 == lane % 4 == w: 32 W is a multiple of 4).
  for (int idx = tid; idx < np * 128; idx += 32 * W) {
    const int pi = idx >> 7, row = (idx & 127) >> 2;
    float accE = 0.0f, accO = 0.0f;
    const float2* abr = ab + pi * nbp * 128 + row * 4 + w;
    const float* d0r = d0s + pi * nbp * 32 + row;
    // Four blocks at a time, the next four loaded while these are chained.
    float2 v[4];
    float dd[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[k] = abr[k * 128];
      dd[k] = d0r[k * 32];
    }
    for (int b0 = 0; b0 < nbp; b0 += 4) {
      float2 vn[4];
      float dn[4];
      const int bn = b0 + 4 < nbp ? b0 + 4 : b0;  // the last round reloads its own blocks
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        vn[k] = abr[(bn + k) * 128];
        dn[k] = d0r[(bn + k) * 32];
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        accE = __fmaf_rn(dd[k], v[k].x, accE);
        accO = __fmaf_rn(dd[k], v[k].y, accO);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[k] = vn[k];
        dd[k] = dn[k];
      }
    }
    const float sum = row_sum(accE, accO);
    const int64_t r = (p0 + pi) * kPanel + row;
    if (w == 0 && r < pr.rows) pr.out[r] = sum;
  }
}

template <class F, int W, int UB, bool MP>
int launch_panel_w(const q1_product* prods, int count, int ppc, cudaStream_t s, const char* who,
                   const L2Ranges& pf) {
  constexpr int PF = 2;
  static bool attr_done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!attr_done[dev]) {
    if (int e = cuda_status(cudaFuncSetAttribute(k_q1_panel<F, W, PF, UB, MP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kPanelSmemMax),
                            "cudaFuncSetAttribute"))
      return e;
    attr_done[dev] = true;
  }
  PanelArgs a = {};
  a.count = count;
  a.ppc = ppc;
  a.pf = pf;
  int ctas = 0, nbp_max = 0;
  for (int j = 0; j < count; ++j) {
    const q1_product& pr = prods[j];
    const Layout L = F::layout(pr.rows, pr.n);
    PanelProd& d = a.p[j];
    d.packed = static_cast<const uint8_t*>(pr.packed);
    d.x = pr.x;
    d.q = pr.q;
    d.d = pr.d;
    d.out = pr.out;
    d.bits_bytes = L.bits_bytes;
    d.rows = int(pr.rows);
    d.nb = int(L.nb);
    d.nbp = int(L.nbp);
    d.panels = int(L.panels);
    d.panel_begin = ctas;
    ctas += (d.panels + ppc - 1) / ppc;
    nbp_max = nbp_max > d.nbp ? nbp_max : d.nbp;
  }
  if (panel_smem_bytes(nbp_max, ppc) > kPanelSmemMax)
    return fail(Q1_ERR_ARG, "%s: %d panels of %d blocks a CTA exceed the shared memory", who, ppc, nbp_max);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(ctas));
  cfg.blockDim = dim3(unsigned(32 * W));
  cfg.dynamicSmemBytes = size_t(panel_smem_bytes(nbp_max, ppc));
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, k_q1_panel<F, W, PF, UB, MP>, a), who);
}

// The kernel's shape for a list of products, or {0, 0}: the most warps W
// (16, 8, 4; starting from the longest row's quads rounded up) whose grid of
// one CTA per panel of every product is one wave; then half-quad units, and
// twice the warps where that still fits, when they lower the work of the
// busiest warp.  When no such shape fits one wave, one CTA of 16 warps per SM
// takes P consecutive panels of a product and builds the activation table
// once for them: the smallest P from ceil(panels / SMs) (at most 8) whose grid
// (ceil(panels_j / P) over the products) is one wave of one CTA per SM and
// whose shared memory fits, with half-quad units when they lower the work of
// the busiest warp (gate and up together: 896 panels, six a CTA).  Failing
// that, a list of two or more products runs one CTA per panel in two waves,
// at the W with the least work per SM; a single product, or more panels than
// two waves, goes to the streaming kernel.
template <class F>
PanelConfig panel_config_for(const q1_product* prods, int count, int sms) {
  if (count < 1 || count > kPanelMaxProducts) return {};
  int64_t panels = 0;
  int nbp = 0;
  for (int j = 0; j < count; ++j) {
    const Layout L = layout_of(prods[j].rows, prods[j].n);
    panels += L.panels;
    nbp = nbp > int(L.nbp) ? nbp : int(L.nbp);
  }
  if (nbp > kPanelMaxNbp) return {};
  const int nq = nbp / 4;
  const int by_smem = kPanelSmemPerSm / (panel_smem_bytes(nbp) + kPanelSmemPerCta);
  auto per_sm = [&](int W) {
    const int by_threads = 2048 / (32 * W);
    int c = panel_ctas_by_regs<F>(W);
    c = c < by_threads ? c : by_threads;
    return c < by_smem ? c : by_smem;
  };
  auto fits = [&](int W) { return panels <= int64_t(per_sm(W)) * sms; };
  auto busiest = [&](int W, int UB) { return (nbp / UB + W - 1) / W * (UB / 2); };  // half quads
  const int W0 = nq > 8 ? 16 : nq > 4 ? 8 : 4;
  int W = 0;
  for (int Wc = W0; Wc >= 4 && !W; Wc >>= 1)
    if (fits(Wc)) W = Wc;
  if (!W) {
    for (int P = int((panels + sms - 1) / sms); P <= kPanelMaxPpc; ++P) {
      if (panel_smem_bytes(nbp, P) > kPanelSmemMax) break;
      int64_t ctas = 0;
      for (int j = 0; j < count; ++j) ctas += (layout_of(prods[j].rows, prods[j].n).panels + P - 1) / P;
      if (ctas > sms) continue;
      const int b4 = (P * nbp / 4 + 15) / 16 * 2, b2 = (P * nbp / 2 + 15) / 16;  // busiest warp's half quads
      return PanelConfig{16, b2 < b4 ? 2 : 4, P};
    }
    if (count < 2) return {};
    int64_t best = 0;
    for (int Wc = W0; Wc >= 4; Wc >>= 1) {
      if (panels > 2 * int64_t(per_sm(Wc)) * sms) continue;
      const int64_t work = (panels + sms - 1) / sms * busiest(Wc, 4) * Wc;  // warp half-quads per SM
      if (!W || work < best) W = Wc, best = work;
    }
    return W ? PanelConfig{W, 4, 1} : PanelConfig{};
  }
  PanelConfig c{W, 4, 1};
  if (busiest(W, 2) < busiest(W, 4)) c.unit = 2;
  if (2 * W <= 16 && fits(2 * W) && busiest(2 * W, 2) < busiest(c.warps, c.unit)) c = PanelConfig{2 * W, 2, 1};
  return c;
}

}  // namespace

template <class F>
PanelConfig panel_config(const q1_product* prods, int count, int sms) {
  return panel_config_for<F>(prods, count, sms);
}
template PanelConfig panel_config<FmtQ1>(const q1_product*, int, int);
template PanelConfig panel_config<FmtQ2>(const q1_product*, int, int);

template <class F>
int launch_panel(const q1_product* prods, int count, PanelConfig c, cudaStream_t s, const char* who,
                 const L2Ranges& pf) {
  if (count < 1 || count > kPanelMaxProducts) return fail(Q1_ERR_ARG, "%s: %d products for the panel kernel", who, count);
  if (c.ppc > 1) {  // several panels a CTA: 16 warps
    switch (c.warps * 10 + c.unit) {
      case 164: return launch_panel_w<F, 16, 4, true>(prods, count, c.ppc, s, who, pf);
      case 162: return launch_panel_w<F, 16, 2, true>(prods, count, c.ppc, s, who, pf);
      default: return fail(Q1_ERR_ARG, "%s: %d warps x %d-block units for %d panels a CTA", who, c.warps, c.unit, c.ppc);
    }
  }
  switch (c.warps * 10 + c.unit) {
    case 164: return launch_panel_w<F, 16, 4, false>(prods, count, 1, s, who, pf);
    case 162: return launch_panel_w<F, 16, 2, false>(prods, count, 1, s, who, pf);
    case 84: return launch_panel_w<F, 8, 4, false>(prods, count, 1, s, who, pf);
    case 82: return launch_panel_w<F, 8, 2, false>(prods, count, 1, s, who, pf);
    case 44: return launch_panel_w<F, 4, 4, false>(prods, count, 1, s, who, pf);
    case 42: return launch_panel_w<F, 4, 2, false>(prods, count, 1, s, who, pf);
    default: return fail(Q1_ERR_ARG, "%s: %d warps x %d-block units per panel", who, c.warps, c.unit);
  }
}
template int launch_panel<FmtQ1>(const q1_product*, int, PanelConfig, cudaStream_t, const char*, const L2Ranges&);
template int launch_panel<FmtQ2>(const q1_product*, int, PanelConfig, cudaStream_t, const char*, const L2Ranges&);

}  // namespace q1
