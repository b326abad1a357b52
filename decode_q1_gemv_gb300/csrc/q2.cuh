// q2.cuh -- the Q2_0 (ternary) format: device layout, activation constants
// and the row-product step.
//
// The pages name Q2_0 as the ternary sibling of Q1_0 and as the next GPU
// kernel (bankML "docs/modules/gpu.md", "Advantages and efficiency" and
// "Limitations") without giving its layout or arithmetic.  This library takes
// the 34-byte block (fp16 scale d0, then 2-bit codes 0/1/2 meaning -1/0/+1)
// and the row product of Q1_0 with ternary lane sums: +1 contributes q, -1 the
// i8 negation of q (-(-128) stays -128), 0 nothing; blocks, sub-blocks, lanes,
// the fma chain and the horizontal sum are Q1_0's.
//
// Device layout: the Q1_0 layout with two sign planes.  For panel group gi,
// quad qd and panel pi, one 4 KB record holds the P words (bit set where the
// weight is +1) in its first 2 KB and the N words (weight -1) in its second,
// each laid out exactly as a Q1_0 quad record (32 rows x 4 words x 4 blocks,
// bit 8*i + pl of word w = element i of lane w (even pl) or w + 4 (odd pl) of
// sub-block pl >> 1).  Scales follow the bits as in Q1_0.
//
// Lane sum.  With a word masked to plane pl (bytes 0 or 2^pl) the exact sum
// is two chained dp4a:
//   dp4a(P_pl, q, dp4a(N_pl, nq, 0x4B400000)),  nq = the bytewise i8 negation
// of q (which wraps -128 to -128 by itself), has the bits of the float
// 1.5*2^23 + 2^pl * s for |2^pl * s| <= 2^16.  With d' = d1 * 2^-pl and
// K = -d' * 1.5*2^23 (both exact), fma(d', that, K) = d1 * s exactly, and the
// chain proceeds as for Q1_0.  The table keeps, per sub-block and word w,
// {q lane w, q lane w+4, nq lane w, nq lane w+4} where Q1_0 keeps its
// accumulator inits, and {d'_even, d'_odd, K_even, K_odd}.
#pragma once

#include "table.cuh"

namespace q1 {

constexpr int kQ2QuadBits = 4096;  // one panel x one quad: P (2 KB) then N (2 KB)

__host__ __device__ __forceinline__ int64_t q2_quad_bits_offset(int64_t p, int64_t qd, int64_t nbp) {
  return (((p / kGroup) * (nbp / 4) + qd) * kGroup + p % kGroup) * kQ2QuadBits;
}
// Word index of (panel p, block b, panel row r, word w) in plane 0 (P) or 1 (N).
__host__ __device__ __forceinline__ int64_t q2_bits_word_index(int64_t p, int64_t b, int r, int w, int64_t nbp,
                                                               int plane) {
  return ((((p / kGroup) * (nbp / 4) + b / 4) * kGroup + p % kGroup) * 2 + plane) * 512 + r * 16 + w * 4 + (b % 4);
}

inline Layout layout_q2(int64_t rows, int64_t n) {
  Layout L = layout_of(rows, n);
  L.bits_bytes = L.rows_pad * L.nbp * 32;
  L.total_bytes = L.bits_bytes + L.scales_bytes;
  return L;
}

struct ConstsQ2 {
  static __device__ __forceinline__ void lane(uint32_t word, int, int, uint32_t& qp, uint32_t& nq) {
    qp = word;
    nq = __vsub4(0u, word);  // per-byte 0 - q modulo 256: -(-128) stays -128
  }
  static __device__ __forceinline__ void lane_no_m128(uint32_t word, int k, int par, uint32_t& qp, uint32_t& nq) {
    lane(word, k, par, qp, nq);
  }
  static __device__ __forceinline__ void scale(float d1, int k, int par, float& dprime, float& K) {
    dprime = __fmul_rn(d1, pow2i(-(2 * k + par)));
    K = -__fmul_rn(dprime, kMagic);
  }
};

// Sub-block K of block BQ of a quad for R rows (P words pv, N words nv):
// ab = d1*s (K = 0) or add.rn(ab, d1*s), lanes w (abE) and w + 4 (abO).
template <int R, int BQ, int K>
__device__ __forceinline__ void q2_quad_subblock(const uint4 (&pv)[R], const uint4 (&nv)[R], const uint4* QCq,
                                                 const float4* DKq, int w, float (&abE)[R], float (&abO)[R]) {
  const uint4 qc = QCq[(BQ * 4 + K) * 4 + w];
  const float4 dk = DKq[BQ * 4 + K];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint32_t P = word_at<BQ>(pv[r]), N = word_at<BQ>(nv[r]);
    const uint32_t even = 0x01010101u << (2 * K), odd = 0x02020202u << (2 * K);
    const uint32_t D0 = dp4a_us(P & even, qc.x, dp4a_us(N & even, qc.z, kMagicBits));
    const uint32_t D1 = dp4a_us(P & odd, qc.y, dp4a_us(N & odd, qc.w, kMagicBits));
    const float pE = __fmaf_rn(dk.x, __uint_as_float(D0), dk.z);
    const float pO = __fmaf_rn(dk.y, __uint_as_float(D1), dk.w);
    if constexpr (K == 0) {
      abE[r] = pE;
      abO[r] = pO;
    } else {
      abE[r] = __fadd_rn(abE[r], pE);
      abO[r] = __fadd_rn(abO[r], pO);
    }
  }
}

template <int R, int BQ>
__device__ __forceinline__ void q2_quad_block(const uint4 (&pv)[R], const uint4 (&nv)[R], const uint2 (&sc)[R],
                                              const uint4* QCq, const float4* DKq, int w, float (&accE)[R],
                                              float (&accO)[R]) {
  float abE[R], abO[R];
  q2_quad_subblock<R, BQ, 0>(pv, nv, QCq, DKq, w, abE, abO);
  q2_quad_subblock<R, BQ, 1>(pv, nv, QCq, DKq, w, abE, abO);
  q2_quad_subblock<R, BQ, 2>(pv, nv, QCq, DKq, w, abE, abO);
  q2_quad_subblock<R, BQ, 3>(pv, nv, QCq, DKq, w, abE, abO);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float d0 = quad_scale<BQ>(sc[r]);
    accE[r] = __fmaf_rn(d0, abE[r], accE[r]);
    accO[r] = __fmaf_rn(d0, abO[r], accO[r]);
  }
}

// A whole quad (4 blocks) for R rows.
template <int R>
__device__ __forceinline__ void q2_quad_all(const uint4 (&pv)[R], const uint4 (&nv)[R], const uint2 (&sc)[R],
                                            const uint4* QCq, const float4* DKq, int w, float (&accE)[R],
                                            float (&accO)[R]) {
  q2_quad_block<R, 0>(pv, nv, sc, QCq, DKq, w, accE, accO);
  q2_quad_block<R, 1>(pv, nv, sc, QCq, DKq, w, accE, accO);
  q2_quad_block<R, 2>(pv, nv, sc, QCq, DKq, w, accE, accO);
  q2_quad_block<R, 3>(pv, nv, sc, QCq, DKq, w, accE, accO);
}

}  // namespace q1
