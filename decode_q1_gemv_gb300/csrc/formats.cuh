// formats.cuh -- the two weight formats as the matrix-vector kernels see
// them.  Q1_0: one sign word per lane word (2 KB per panel and quad, layout in
// common.cuh).  Q2_0: a P and an N word (4 KB), see q2.cuh.
#pragma once

#include "q2.cuh"

namespace q1 {

struct FmtQ1 {
  static constexpr int kQuadBits = 2048;  // one panel x one quad of blocks: 32 rows x 4 blocks x 16 B
  static constexpr bool kTwoPlanes = false;
  static constexpr int kBigRows = 8;      // rows per thread of the streaming launches that fill every CTA
  using Consts = ConstsQ1;
  static __host__ __device__ __forceinline__ int64_t quad_bits_offset(int64_t p, int64_t qd, int64_t nbp) {
    return q1::quad_bits_offset(p, qd, nbp);
  }
  static Layout layout(int64_t rows, int64_t n) { return layout_of(rows, n); }
};
struct FmtQ2 {
  static constexpr int kQuadBits = kQ2QuadBits;
  static constexpr bool kTwoPlanes = true;
  static constexpr int kBigRows = 8;      // 168 registers, no spills; 4 rows x 2 slots measured 0.7 % slower
  using Consts = ConstsQ2;
  static __host__ __device__ __forceinline__ int64_t quad_bits_offset(int64_t p, int64_t qd, int64_t nbp) {
    return q2_quad_bits_offset(p, qd, nbp);
  }
  static Layout layout(int64_t rows, int64_t n) { return layout_q2(rows, n); }
};

// panel.cu: the kernel for launches of few rows in total (one CTA per panel
// of each of up to 8 products).  panel_config: its shape for a product list
// (warps per CTA, blocks per work unit), {0, 0} when the streaming kernel
// serves it (more than 8 products, a row too long for the CTA's shared
// memory, or more panels than one wave of CTAs).
struct PanelConfig {
  int warps = 0;  // W: 16, 8 or 4
  int unit = 0;   // blocks per work unit: 4 (a quad) or 2 (half a quad)
  int ppc = 1;    // consecutive panels of a product per CTA
};
template <class F>
PanelConfig panel_config(const q1_product* prods, int count, int sms);
template <class F>
int launch_panel(const q1_product* prods, int count, PanelConfig c, cudaStream_t s, const char* who,
                 const L2Ranges& pf);

}  // namespace q1
