// multi.cu -- the streaming matrix-vector kernel behind q1_0_gemv_multi /
// q2_0_gemv_multi (up to Q1_MAX_PRODUCTS independent products in one launch)
// and q1_0_gemv / q2_0_gemv, for launches of many rows or many products; the
// launcher here (launch_products) sends launches of a few thousand rows in
// total to the panel kernel (panel.cu) instead.
//
// Definition (bankML "docs/modules/gpu.md", "kernels.rs -- the Q1_0 kernels",
// first and second bullets): each output row is one dot product of 128-weight
// blocks, four sub-blocks each, eight lanes of exact integer sums (i8 negation
// wraps -128 to -128), ab = d1*s then fma(d1, s, ab), acc = fma(d0, ab, acc),
// and the horizontal sum (a0+a4 + a2+a6) + (a1+a5 + a3+a7).  Lanes are
// independent chains, so four threads share a row, two lanes each; table.cuh
// explains how every step keeps the definition's single roundings, and q2.cuh
// the same for the ternary Q2_0 format (the kernel is a template over the
// format: FmtQ1, FmtQ2).
//
// Structure.  A CTA is one producer warp and four consumer warps per panel
// slot (two slots for R <= 2 rows per thread, one for R = 8).  The producer
// streams packed weights HBM -> shared memory with 1-D bulk copies into a
// ring of stages (mbarrier full/empty pairs).  A stage is one quad of blocks
// (4 x 128 weights per row) for the CTA's current tile of slots*R panels (8
// panels = 256 rows for the large launches): 2 KB (Q2_0: 4 KB) of sign words
// and 256 B of scales per panel, two contiguous copies thanks to the packed
// layout.  Consumer thread (row, lane pair) handles R rows of a tile.  CTAs
// are persistent: the products' tiles lie on one cost axis, each CTA owns a
// contiguous range of it (placed by the host for many-product launches) and
// starts at its first product by binary search; the producer runs ahead
// across tile and product boundaries.  The producer reads only weights, so it
// starts before griddepcontrol.wait; consumers wait for the preceding kernel
// before reading the activation (f32, quantized here exactly as
// q8_quantize_act does, or already quantized).  Every wait is bounded and
// reports through the device status word instead of hanging.
#include <algorithm>

#include "formats.cuh"

namespace q1 {

static __device__ unsigned g_status_dp4a = 0u;

// Panels computed side by side (4 consumer warps = 32 rows each): two for
// R <= 2 rows per thread, one for R = 8 (an 8-panel tile with half the warps
// of two slots of four rows, which measured slower).
template <int R>
__host__ __device__ constexpr int slots_of() { return R >= 8 ? 1 : 2; }
template <int R>
__host__ __device__ constexpr int consumer_warps() { return 4 * slots_of<R>(); }
template <int R>
__host__ __device__ constexpr int consumers() { return 32 * consumer_warps<R>(); }
template <int R>
__host__ __device__ constexpr int multi_threads() { return consumers<R>() + 32; }
constexpr int kQuadScales = 256;   // 32 rows x 4 blocks x 2 B

constexpr int kConsumerBarrier = 1;
constexpr int kMaxKc = 128;        // blocks of activation held in the table (n <= 16384 in one chunk)

struct MProd {
  const uint8_t* packed;
  const float* x;        // f32 activation, or null
  const int8_t* q;       // q8_0 quants (when x is null)
  const uint16_t* d;     // q8_0 scales (when x is null)
  float* out;
  int64_t bits_bytes;
  int64_t cost_begin;    // sum over earlier products of tiles * nbp
  int rows, nb, nbp, panels, tiles;
};

constexpr int kMaxCuts = 512;  // CTAs of a many-product launch that get host-computed ranges

template <int PMAX>
struct MArgs {
  MProd p[PMAX];
  int64_t total_cost;
  int count;
  int kc;                // table chunk in blocks (multiple of 4)
  int ncut;              // 0: equal split of the cost axis; else CTA b owns [cut[b], cut[b+1])
  L2Ranges pf;           // pulled into L2 while this launch runs (the next launch's inputs)
  int64_t cut[PMAX > 8 ? kMaxCuts + 1 : 1];
};

// Ring of stages: a stage is one quad of blocks for the tile's slots*R panels;
// about 72 KB of weights in flight per CTA (at least two stages).
template <int R, class F>
__host__ __device__ constexpr int stage_bytes() { return slots_of<R>() * R * (F::kQuadBits + kQuadScales); }
template <int R, class F>
__host__ __device__ constexpr int ring_stages() {
  return 73728 / stage_bytes<R, F>() > 2 ? 73728 / stage_bytes<R, F>() : 2;
}

template <int R, class F>
__host__ __device__ constexpr int multi_smem_bytes(int kc) {
  return ring_stages<R, F>() * stage_bytes<R, F>() + table_bytes(kc) + 2 * ring_stages<R, F>() * 8;
}

// Tiles [t_lo, t_hi) of product p that fall in this CTA's cost range.
__host__ __device__ __forceinline__ void tile_range(const MProd& p, int64_t lo, int64_t hi, int& t_lo, int& t_hi) {
  const int64_t c = p.nbp;
  auto first_at_or_after = [&](int64_t v) -> int {
    int64_t t = v <= p.cost_begin ? 0 : (v - p.cost_begin + c - 1) / c;
    return int(t < p.tiles ? t : p.tiles);
  };
  t_lo = first_at_or_after(lo);
  t_hi = first_at_or_after(hi);
}

// The product holding cost v: the last one whose first tile's cost is <= v
// (cost_begin strictly increases, every product having at least one tile).
// A CTA starts its walk there instead of scanning every earlier product: each
// tile_range costs two 64-bit divisions, and a scan over a couple of hundred
// products delayed the last CTAs of a launch by tens of microseconds.
template <int PMAX>
__device__ __forceinline__ int first_product(const MArgs<PMAX>& a, int64_t v) {
  int l = 0, h = a.count;
  while (h - l > 1) {
    const int m = (l + h) >> 1;
    if (a.p[m].cost_begin <= v) l = m; else h = m;
  }
  return l;
}

template <int R, int PMAX, class F>
__global__ void __launch_bounds__(multi_threads<R>(), 2) k_q1_multi(const __grid_constant__ MArgs<PMAX> a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int S = ring_stages<R, F>();
  constexpr int SB = stage_bytes<R, F>();
  constexpr int kSlots = slots_of<R>();
  constexpr int kConsumerWarps = consumer_warps<R>();
  constexpr int kConsumers = consumers<R>();
  constexpr int TB = kSlots * R * F::kQuadBits;  // bits part of a stage
  constexpr int kTableBatch = R >= 8 ? 8 : 4;  // load rounds in flight while a table is built
  constexpr int kTableBatchX = R >= 8 ? 4 : R >= 2 ? 2 : 1;  // the same from f32 (two words a round)
  unsigned char* table = smem + S * SB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(table + table_bytes(a.kc));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t lo = a.total_cost * int64_t(blockIdx.x) / int64_t(gridDim.x);
  int64_t hi = a.total_cost * int64_t(blockIdx.x + 1) / int64_t(gridDim.x);
  if constexpr (PMAX > 8) {
    if (a.ncut) {
      lo = a.cut[blockIdx.x];
      hi = a.cut[blockIdx.x + 1];
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&bars[s]), 1);
      mbar_init(smem_addr(&bars[S + s]), kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      l2_prefetch_share(a.pf, int(blockIdx.x), int(gridDim.x));  // the next launch's inputs, if given
      bool ok = true;
      int it = 0;
      for (int j = first_product(a, lo); j < a.count && a.p[j].cost_begin < hi && ok; ++j) {
        int t_lo, t_hi;
        tile_range(a.p[j], lo, hi, t_lo, t_hi);
        const uint8_t* bits = a.p[j].packed;
        const uint8_t* scales = bits + a.p[j].bits_bytes;
        const int nbp = a.p[j].nbp;
        const int quads = nbp / 4;
        for (int t = t_lo; t < t_hi && ok; ++t) {
          const int64_t p0 = int64_t(t) * kSlots * R;  // aligned panels inside one panel group
          for (int qd = 0; qd < quads; ++qd, ++it) {
            const int s = it % S;
            if (it >= S && !mbar_wait(smem_addr(&bars[S + s]), uint32_t(it / S - 1) & 1u)) {
              ok = false;
              break;
            }
            const uint32_t full = smem_addr(&bars[s]);
            mbar_arrive_expect_tx(full, uint32_t(SB));
            const uint32_t dst = smem_addr(smem + s * SB);
            bulk_g2s(dst, bits + F::quad_bits_offset(p0, qd, nbp), TB, full);
            bulk_g2s(dst + TB, scales + quad_scales_offset(p0, qd, nbp), kSlots * R * kQuadScales, full);
          }
        }
      }
      if (!ok) atomicOr(&g_status_dp4a, kStatusWaitTimeout);
      // The CTA's shared memory must outlive every copy issued into it: wait
      // (bounded) until the last S stages have landed.  On the normal path the
      // consumers have already waited for them and this returns at once.
      for (int k = it > S ? it - S : 0; k < it; ++k)
        mbar_wait(smem_addr(&bars[k % S]), uint32_t(k / S) & 1u, 100000000ull);
    }
    return;
  }

  // ------------------------------- consumers ------------------------------
  const int tid = threadIdx.x;
  const int ps = warp >> 2;                       // panel slot within the tile
  const int prow = (warp & 3) * 8 + (lane >> 2);  // row within the panel
  const int w = lane & 3;                         // word w: lanes w and w+4
  const uint4* QC = reinterpret_cast<const uint4*>(table);
  const float4* DK = reinterpret_cast<const float4*>(table + table_dk_offset(a.kc));
  const int kc = a.kc;

  pdl_wait();  // the activations may be written by the preceding kernel

  // Last tile of this CTA (dependents are signalled when it starts).
  int last_j = -1, last_t = -1;
  const int j_first = first_product(a, lo);
  for (int j = j_first; j < a.count && a.p[j].cost_begin < hi; ++j) {
    int t_lo, t_hi;
    tile_range(a.p[j], lo, hi, t_lo, t_hi);
    if (t_lo < t_hi) {
      last_j = j;
      last_t = t_hi - 1;
    }
  }
  if (last_j < 0) pdl_launch_dependents();

  // A consumer wait can only give up on a stage whose copy never lands.  Every
  // consumer warp needs that stage before its next named barrier, so all of
  // them give up at the same stage and leave without reaching a barrier the
  // others wait at; the lanes of a warp poll the same barrier and clock in
  // step, so they decide together.
  bool ok = true;
  int it = 0;
  for (int j = j_first; j < a.count && a.p[j].cost_begin < hi && ok; ++j) {
    int t_lo, t_hi;
    tile_range(a.p[j], lo, hi, t_lo, t_hi);
    if (t_lo >= t_hi) continue;
    const float* px = a.p[j].x;
    const int8_t* pq = a.p[j].q;
    const uint16_t* pd = a.p[j].d;
    float* pout = a.p[j].out;
    const int prows = a.p[j].rows, pnb = a.p[j].nb, pnbp = a.p[j].nbp;
    const int quads = pnbp / 4;
    const bool one_chunk = pnbp <= kc;
    if (one_chunk) {
      named_barrier(kConsumerBarrier, kConsumers);  // previous product's table no longer read
      if (px) build_table_x<kTableBatchX, typename F::Consts>(px, pnb, 0, pnbp, table, tid, kConsumers, kc);
      else build_table_q<kTableBatch, typename F::Consts>(pq, pd, pnb, 0, pnbp, table, tid, kConsumers, kc);
      named_barrier(kConsumerBarrier, kConsumers);
    }
    for (int t = t_lo; t < t_hi && ok; ++t) {
      if (j == last_j && t == last_t) pdl_launch_dependents();
      float accE[R], accO[R];
#pragma unroll
      for (int r = 0; r < R; ++r) accE[r] = accO[r] = 0.0f;

      for (int qd = 0; qd < quads; ++qd, ++it) {
        const int b0 = qd * 4;
        if (!one_chunk && b0 % kc == 0) {
          named_barrier(kConsumerBarrier, kConsumers);
          const int kcb = min(kc, pnbp - b0);
          if (px) build_table_x<kTableBatchX, typename F::Consts>(px, pnb, b0, kcb, table, tid, kConsumers, kc);
          else build_table_q<kTableBatch, typename F::Consts>(pq, pd, pnb, b0, kcb, table, tid, kConsumers, kc);
          named_barrier(kConsumerBarrier, kConsumers);
        }
        const int gb = one_chunk ? b0 : b0 % kc;  // block index within the table
        const int s = it % S;
        if (!mbar_wait(smem_addr(&bars[s]), uint32_t(it / S) & 1u)) {
          ok = false;
          break;
        }
        const unsigned char* st = smem + s * SB;
        uint4 wv[R], nv[F::kTwoPlanes ? R : 1];
        uint2 sc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int tp = kSlots * r + ps;
          wv[r] = reinterpret_cast<const uint4*>(st + tp * F::kQuadBits)[prow * 4 + w];
          if constexpr (F::kTwoPlanes) nv[r] = reinterpret_cast<const uint4*>(st + tp * F::kQuadBits + 2048)[prow * 4 + w];
          sc[r] = reinterpret_cast<const uint2*>(st + TB + tp * kQuadScales)[prow];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bars[S + s]));  // stage consumed

        if constexpr (F::kTwoPlanes) q2_quad_all<R>(wv, nv, sc, QC + gb * 16, DK + gb * 4, w, accE, accO);
        else quad_all<R>(wv, sc, QC + gb * 16, DK + gb * 4, w, accE, accO);
      }
      if (!ok) break;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float sum = row_sum(accE[r], accO[r]);
        const int64_t row = (int64_t(t) * kSlots * R + kSlots * r + ps) * kPanel + prow;
        if (w == 0 && row < prows) pout[row] = sum;
      }
    }
  }
  if (!ok) atomicOr(&g_status_dp4a, kStatusWaitTimeout);
}

// ---------------------------------------------------------------- host ----
template <int R, int PMAX, class F>
static int set_smem_attr() {
  static int done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_q1_multi<R, PMAX, F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         multi_smem_bytes<R, F>(kMaxKc));
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute");
    done[dev] = 1;
  }
  return Q1_OK;
}

// Cuts of the cost axis at tile boundaries for at most G contiguous ranges
// whose largest cost is at most V, filled greedily in product order; false if
// V does not suffice.  cut[0..nseg] receives the boundaries when non-null.
template <int PMAX>
static bool fill_ranges(const MArgs<PMAX>& a, int64_t V, int G, int64_t* cut, int& nseg) {
  int seg = 0;
  int64_t cur = 0, pos = 0;
  if (cut) cut[0] = 0;
  for (int j = 0; j < a.count; ++j) {
    const int64_t c = a.p[j].nbp;
    if (c > V) return false;
    int64_t left = a.p[j].tiles;
    while (left > 0) {
      const int64_t k = std::min(left, (V - cur) / c);
      if (k == 0) {
        if (++seg >= G) return false;
        if (cut) cut[seg] = pos;
        cur = 0;
        continue;
      }
      cur += k * c;
      pos += k * c;
      left -= k;
    }
  }
  nseg = seg + 1;
  if (cut) cut[nseg] = pos;
  return true;
}

// G contiguous ranges, none above V, each aiming at the average of what is
// left (the boundary goes to the nearer tile edge), so that every CTA gets
// work even when the greedy fill at V would need fewer ranges; false if tiles
// remain after G ranges.
template <int PMAX>
static bool fill_even(const MArgs<PMAX>& a, int64_t V, int G, int64_t* cut) {
  int j = 0;
  int64_t left = a.count > 0 ? a.p[0].tiles : 0, pos = 0;
  cut[0] = 0;
  for (int seg = 0; seg < G; ++seg) {
    const int64_t target = (a.total_cost - pos + (G - seg) - 1) / (G - seg);
    int64_t cur = 0;
    while (j < a.count) {
      if (left == 0) {
        if (++j < a.count) left = a.p[j].tiles;
        continue;
      }
      if (cur >= target) break;
      const int64_t c = a.p[j].nbp;
      int64_t k = std::min(left, std::min((V - cur) / c, (target - cur) / c));  // >= 0
      // one tile past the target when that lands nearer to it, within V
      if (k < left && cur + (k + 1) * c <= V && (cur + k * c == 0 || cur + (k + 1) * c - target < target - cur - k * c))
        ++k;
      cur += k * c;
      pos += k * c;
      left -= k;
      if (left > 0) break;  // the range ends inside product j
    }
    cut[seg + 1] = pos;
  }
  return pos == a.total_cost;
}

// The smallest largest-range cost V for G contiguous ranges: the equal share
// rounded up always fits once a whole tile is added, so V is searched in
// [share, share + largest tile cost].  The ranges are then spread over all G
// CTAs (fill_even), or, if that does not close, kept as the greedy fill made
// them.
template <int PMAX>
static int balanced_ranges(MArgs<PMAX>& a, int G, int64_t max_tile) {
  int64_t lo = (a.total_cost + G - 1) / G, hi = lo + max_tile;
  int nseg = 0;
  while (lo < hi) {
    const int64_t m = (lo + hi) / 2;
    if (fill_ranges(a, m, G, nullptr, nseg)) hi = m;
    else lo = m + 1;
  }
  if (fill_even(a, lo, G, a.cut)) {
    nseg = G;
  } else {
    fill_ranges(a, lo, G, a.cut, nseg);
  }
  a.ncut = nseg;
  return nseg;
}

// The launch plan of k_q1_multi<R, PMAX> for `count` products on `sms` SMs:
// the kernel arguments and the grid.
template <int R, int PMAX, class F>
static void plan_multi(const q1_product* prods, int count, int sms, MArgs<PMAX>& a, int& grid) {
  int64_t cost = 0;
  int64_t total_tiles = 0;
  int max_nbp = 8;
  for (int j = 0; j < count; ++j) {
    const Layout L = F::layout(prods[j].rows, prods[j].n);
    MProd& p = a.p[j];
    p.packed = static_cast<const uint8_t*>(prods[j].packed);
    p.x = prods[j].x;
    p.q = prods[j].q;
    p.d = prods[j].d;
    p.out = prods[j].out;
    p.bits_bytes = L.bits_bytes;
    p.rows = int(L.rows);
    p.nb = int(L.nb);
    p.nbp = int(L.nbp);
    p.panels = int(L.panels);
    p.tiles = int(L.panels / (slots_of<R>() * R));  // panels come in groups of 8, so tiles are whole
    p.cost_begin = cost;
    cost += int64_t(p.tiles) * p.nbp;
    total_tiles += p.tiles;
    max_nbp = std::max(max_nbp, p.nbp);
  }
  a.total_cost = cost;
  a.count = count;
  a.kc = std::min(max_nbp, kMaxKc);
  a.ncut = 0;
  grid = int(std::min<int64_t>(total_tiles, 2 * int64_t(sms)));
  // Many products of unequal tile costs: an equal split of the cost axis,
  // rounded to whole tiles, leaves up to a tile's cost of imbalance per CTA;
  // the host places the boundaries so that the largest range is as small as
  // contiguous ranges allow.
  if constexpr (PMAX > 8) {
    if (grid <= kMaxCuts) grid = balanced_ranges(a, grid, max_nbp);
  }
}

template <int R, int PMAX, class F>
static int launch_multi(const q1_product* prods, int count, cudaStream_t s, const char* who, const L2Ranges& pf) {
  if (int e = set_smem_attr<R, PMAX, F>()) return e;
  MArgs<PMAX> a;
  int grid = 0;
  plan_multi<R, PMAX, F>(prods, count, num_sms(), a, grid);
  a.pf = pf;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(multi_threads<R>());
  cfg.dynamicSmemBytes = size_t(multi_smem_bytes<R, F>(a.kc));
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, k_q1_multi<R, PMAX, F>, a), who);
}

// The plan reported by q1_0_gemv_multi_plan: the CTA ranges exactly as the
// kernel derives them from the arguments, and their tile costs.
template <int R, int PMAX, class F>
static int report_plan(const q1_product* prods, int count, int sms, q1_multi_plan* out, int64_t* cuts,
                       int max_cuts) {
  MArgs<PMAX>* a = new MArgs<PMAX>;
  int grid = 0;
  plan_multi<R, PMAX, F>(prods, count, sms, *a, grid);
  out->rows_per_thread = R;
  out->panel_warps = 0;
  out->panel_unit_blocks = 0;
  out->panel_panels = 0;
  out->grid = grid;
  out->total_cost = a->total_cost;
  out->max_range_cost = 0;
  for (int b = 0; b < grid; ++b) {
    int64_t lo = a->total_cost * b / grid, hi = a->total_cost * (b + 1) / grid;
    if (a->ncut) {
      lo = a->cut[b];
      hi = a->cut[b + 1];
    }
    int64_t c = 0;
    for (int j = 0; j < count; ++j) {
      int t_lo, t_hi;
      tile_range(a->p[j], lo, hi, t_lo, t_hi);
      c += int64_t(t_hi - t_lo) * a->p[j].nbp;
    }
    out->max_range_cost = std::max(out->max_range_cost, c);
    if (cuts && b < max_cuts) cuts[b] = lo;
    if (cuts && b + 1 < max_cuts && b == grid - 1) cuts[b + 1] = hi;
  }
  delete a;
  return Q1_OK;
}

// Rows per thread: the largest R whose tiles still give every CTA some work
// (the 8-panel tiles take the format's big-launch rows per thread).
template <class F>
static int rows_per_thread(const q1_product* prods, int count, int sms) {
  int64_t panels = 0;
  for (int j = 0; j < count; ++j) panels += (prods[j].rows + kPanel - 1) / kPanel;
  const int64_t ctas = 2 * int64_t(sms);
  return panels >= 8 * ctas ? F::kBigRows : panels >= 4 * ctas ? 2 : 1;
}

template <int PMAX, class F>
static int dispatch(const q1_product* prods, int count, cudaStream_t s, const char* who, const L2Ranges& pf) {
  switch (rows_per_thread<F>(prods, count, num_sms())) {
    case F::kBigRows: return launch_multi<F::kBigRows, PMAX, F>(prods, count, s, who, pf);
    case 2: return launch_multi<2, PMAX, F>(prods, count, s, who, pf);
    default: return launch_multi<1, PMAX, F>(prods, count, s, who, pf);
  }
}

template <int PMAX, class F>
static int dispatch_plan(const q1_product* prods, int count, int sms, q1_multi_plan* out, int64_t* cuts,
                         int max_cuts) {
  switch (rows_per_thread<F>(prods, count, sms)) {
    case F::kBigRows: return report_plan<F::kBigRows, PMAX, F>(prods, count, sms, out, cuts, max_cuts);
    case 2: return report_plan<2, PMAX, F>(prods, count, sms, out, cuts, max_cuts);
    default: return report_plan<1, PMAX, F>(prods, count, sms, out, cuts, max_cuts);
  }
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int v = 0;
    cached[dev] = (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) ? v : 148;
  }
  return cached[dev];
}

int check_product(const char* who, int idx, const q1_product& pr) {
  if (pr.rows < 1 || pr.rows > (int64_t(1) << 26) || pr.n < 128 || pr.n > (int64_t(1) << 24) || pr.n % 128)
    return fail(Q1_ERR_ARG, "%s: product %d: bad shape rows=%lld n=%lld", who, idx, (long long)pr.rows,
                (long long)pr.n);
  if (!pr.packed || !pr.out || (!pr.x && (!pr.q || !pr.d)))
    return fail(Q1_ERR_ARG, "%s: product %d: null pointer", who, idx);
  auto mis = [](const void* p) { return p && reinterpret_cast<uintptr_t>(p) % 16 != 0; };
  if (mis(pr.packed) || mis(pr.x) || mis(pr.q) || mis(pr.d) || mis(pr.out))
    return fail(Q1_ERR_ARG, "%s: product %d: buffers must be 16-byte aligned", who, idx);
  return Q1_OK;
}

template <class F>
static int launch_products(const q1_product* prods, int count, cudaStream_t s, const char* who,
                           const L2Ranges& pf = L2Ranges{}) {
  const PanelConfig c = panel_config<F>(prods, count, num_sms());
  if (c.warps) return launch_panel<F>(prods, count, c, s, who, pf);
  if (count == 1) return dispatch<1, F>(prods, count, s, who, pf);
  if (count <= 8) return dispatch<8, F>(prods, count, s, who, pf);
  return dispatch<Q1_MAX_PRODUCTS, F>(prods, count, s, who, pf);
}

int launch_products_dp4a(const q1_product* prods, int count, cudaStream_t s, const char* who, const L2Ranges& pf) {
  return launch_products<FmtQ1>(prods, count, s, who, pf);
}

int status_word_dp4a(unsigned* v, int clear) {
  if (int e = cuda_status(cudaMemcpyFromSymbol(v, g_status_dp4a, sizeof *v), "q1_device_status")) return e;
  if (clear && *v) {
    const unsigned zero = 0;
    return cuda_status(cudaMemcpyToSymbol(g_status_dp4a, &zero, sizeof zero), "q1_device_status");
  }
  return Q1_OK;
}

}  // namespace q1

using namespace q1;

extern "C" int q1_0_gemv(const void* packed, int64_t rows, int64_t n, const int8_t* q, const uint16_t* d,
                         float* out, void* stream) {
  q1_product p = {packed, rows, n, nullptr, q, d, out};
  if (!q || !d) return fail(Q1_ERR_ARG, "q1_0_gemv: null pointer");
  if (int e = check_product("q1_0_gemv", 0, p)) return e;
  return launch_products_dp4a(&p, 1, static_cast<cudaStream_t>(stream), "q1_0_gemv launch");
}

template <class F>
static int multi_plan(const char* who, const q1_product* products, int count, int sms, q1_multi_plan* plan,
                      int64_t* cuts, int max_cuts) {
  if (!products || !plan || count < 1 || count > Q1_MAX_PRODUCTS)
    return fail(Q1_ERR_ARG, "%s: count=%d outside 1..%d (or null list/plan)", who, count, Q1_MAX_PRODUCTS);
  if (sms < 0 || sms > 4096) return fail(Q1_ERR_ARG, "%s: sms=%d outside 0..4096", who, sms);
  for (int j = 0; j < count; ++j) {
    const q1_product& pr = products[j];
    if (pr.rows < 1 || pr.rows > (int64_t(1) << 26) || pr.n < 128 || pr.n > (int64_t(1) << 24) || pr.n % 128)
      return fail(Q1_ERR_ARG, "%s: product %d: bad shape rows=%lld n=%lld", who, j, (long long)pr.rows,
                  (long long)pr.n);
  }
  if (cuts && max_cuts < 0) return fail(Q1_ERR_ARG, "%s: max_cuts=%d < 0", who, max_cuts);
  const int n_sms = sms > 0 ? sms : num_sms();
  const PanelConfig c = panel_config<F>(products, count, n_sms);
  if (c.warps) {
    int64_t ctas = 0;
    for (int j = 0; j < count; ++j) ctas += (F::layout(products[j].rows, products[j].n).panels + c.ppc - 1) / c.ppc;
    plan->rows_per_thread = 4;
    plan->grid = int(ctas);
    plan->total_cost = 0;
    plan->max_range_cost = 0;
    plan->panel_warps = c.warps;
    plan->panel_unit_blocks = c.unit;
    plan->panel_panels = c.ppc;
    return Q1_OK;
  }
  if (count == 1) return dispatch_plan<1, F>(products, count, n_sms, plan, cuts, max_cuts);
  if (count <= 8) return dispatch_plan<8, F>(products, count, n_sms, plan, cuts, max_cuts);
  return dispatch_plan<Q1_MAX_PRODUCTS, F>(products, count, n_sms, plan, cuts, max_cuts);
}

extern "C" int q1_0_gemv_multi_plan(const q1_product* products, int count, int sms, q1_multi_plan* plan,
                                    int64_t* cuts, int max_cuts) {
  return multi_plan<FmtQ1>("q1_0_gemv_multi_plan", products, count, sms, plan, cuts, max_cuts);
}

extern "C" int q2_0_gemv_multi_plan(const q1_product* products, int count, int sms, q1_multi_plan* plan,
                                    int64_t* cuts, int max_cuts) {
  return multi_plan<FmtQ2>("q2_0_gemv_multi_plan", products, count, sms, plan, cuts, max_cuts);
}

extern "C" int q1_0_gemv_multi(const q1_product* products, int count, void* stream) {
  if (!products || count < 1 || count > Q1_MAX_PRODUCTS)
    return fail(Q1_ERR_ARG, "q1_0_gemv_multi: count=%d outside 1..%d (or null list)", count, Q1_MAX_PRODUCTS);
  for (int j = 0; j < count; ++j)
    if (int e = check_product("q1_0_gemv_multi", j, products[j])) return e;
  return launch_products_dp4a(products, count, static_cast<cudaStream_t>(stream), "q1_0_gemv_multi launch");
}

// q1_0_gemv_multi / q2_0_gemv_multi with L2 prefetches of the given ranges,
// issued by the launch's CTAs before they wait for the preceding kernel.
template <class F>
static int multi_prefetch(const char* who, const q1_product* products, int count, const q1_range* prefetch,
                          int nranges, void* stream) {
  if (!products || count < 1 || count > Q1_MAX_PRODUCTS)
    return fail(Q1_ERR_ARG, "%s: count=%d outside 1..%d (or null list)", who, count, Q1_MAX_PRODUCTS);
  for (int j = 0; j < count; ++j)
    if (int e = check_product(who, j, products[j])) return e;
  if (nranges < 0 || nranges > Q1_MAX_PREFETCH_RANGES || (nranges > 0 && !prefetch))
    return fail(Q1_ERR_ARG, "%s: %d prefetch ranges (0..%d)", who, nranges, Q1_MAX_PREFETCH_RANGES);
  L2Ranges pf{};
  for (int i = 0; i < nranges; ++i) {
    const q1_range& r = prefetch[i];
    if (r.bytes < 0 || r.bytes > (int64_t(1) << 40) || (r.bytes > 0 && !r.ptr))
      return fail(Q1_ERR_ARG, "%s: prefetch range %d: %lld bytes at %p", who, i, (long long)r.bytes, r.ptr);
    if (reinterpret_cast<uintptr_t>(r.ptr) % 16 != 0)
      return fail(Q1_ERR_ARG, "%s: prefetch range %d must start 16-byte aligned", who, i);
    if (r.bytes >= 16) pf.r[pf.count++] = L2Range{static_cast<const uint8_t*>(r.ptr), r.bytes / 16 * 16};
  }
  return launch_products<F>(products, count, static_cast<cudaStream_t>(stream), who, pf);
}

extern "C" int q1_0_gemv_multi_prefetch(const q1_product* products, int count, const q1_range* prefetch,
                                        int nranges, void* stream) {
  return multi_prefetch<FmtQ1>("q1_0_gemv_multi_prefetch", products, count, prefetch, nranges, stream);
}

extern "C" int q2_0_gemv_multi_prefetch(const q1_product* products, int count, const q1_range* prefetch,
                                        int nranges, void* stream) {
  return multi_prefetch<FmtQ2>("q2_0_gemv_multi_prefetch", products, count, prefetch, nranges, stream);
}

extern "C" int q2_0_gemv(const void* packed, int64_t rows, int64_t n, const int8_t* q, const uint16_t* d,
                         float* out, void* stream) {
  q1_product p = {packed, rows, n, nullptr, q, d, out};
  if (!q || !d) return fail(Q1_ERR_ARG, "q2_0_gemv: null pointer");
  if (int e = check_product("q2_0_gemv", 0, p)) return e;
  return launch_products<FmtQ2>(&p, 1, static_cast<cudaStream_t>(stream), "q2_0_gemv launch");
}

extern "C" int q2_0_gemv_multi(const q1_product* products, int count, void* stream) {
  if (!products || count < 1 || count > Q1_MAX_PRODUCTS)
    return fail(Q1_ERR_ARG, "q2_0_gemv_multi: count=%d outside 1..%d (or null list)", count, Q1_MAX_PRODUCTS);
  for (int j = 0; j < count; ++j)
    if (int e = check_product("q2_0_gemv_multi", j, products[j])) return e;
  return launch_products<FmtQ2>(products, count, static_cast<cudaStream_t>(stream), "q2_0_gemv_multi launch");
}
