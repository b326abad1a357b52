// table.cuh -- activation-side constants of the Q1_0 x q8_0 row product, kept
// in shared memory by the product kernels.
//
// For every 32-element sub-block g of the activation and lane l (elements
// 4l..4l+3 of the sub-block):
//   q'  = the four int8 quants with -128 replaced by 0 (one 32-bit word)
//   A   = sum(q') + 128 * #(-128)      so that the lane sum is s = 2*M - A
//         with M = sum(bit_i * q'_i) (an i8 negation of -128 stays -128)
//   ci  = 0x4B400000 - 2^(pe-1) * A    dp4a accumulator init, pe = the lane's
//                                      effective bit plane (below)
// and for every sub-block and lane parity
//   d'  = d1 * 2^(1-pe),  K = -d' * 1.5*2^23
// with d1 the sub-block's fp16 scale widened to f32.  Then, for a weight word
// masked to the lane's plane, dp4a(mask, q', ci) has the bits of the float
// F = 1.5*2^23 + 2^(pe-1)*s, and fma(d', F, K) = d1*s exactly.
//
// Layout for a chunk of kc blocks (kc*4 sub-blocks), 80 bytes per sub-block:
//   QC[g][w] (uint4)  = { q' lane w, q' lane w+4, ci lane w, ci lane w+4 }
//   DK[g]    (float4) = { d' lanes 0-3, d' lanes 4-7, K lanes 0-3, K lanes 4-7 }
#pragma once

#include "common.cuh"

namespace q1 {

__host__ __device__ constexpr int table_bytes(int kc) { return kc * 4 * (4 * 16 + 16); }
__host__ __device__ constexpr int table_dk_offset(int kc) { return kc * 4 * 64; }

__device__ __forceinline__ float pow2i(int e) {  // exact 2^e for -126 <= e <= 127
  return __int_as_float((127 + e) << 23);
}

// Effective bit plane of sub-block k for the low (par 0: lanes 0-3, plane 2k)
// or high (par 1: lanes 4-7, plane 2k+1) half of a word.  Plane 0 is used
// shifted left by one (byte values 0/2), so every lane's dp4a result is
// 2^pe * M with pe >= 1 and the activation term enters as 2^(pe-1) * A.
__device__ __forceinline__ int pe_of(int k, int par) { return (k == 0 && par == 0) ? 1 : 2 * k + par; }

__device__ __forceinline__ void lane_consts(uint32_t word, int k, int par, uint32_t& qp, uint32_t& ci) {
  const uint32_t m80 = __vcmpeq4(word, 0x80808080u);  // 0xff in bytes equal to -128
  qp = word & ~m80;
  const int cnt = __popc(m80) >> 3;
  const int A = __dp4a(int(qp), 0x01010101, 0) + 128 * cnt;
  ci = uint32_t(int(kMagicBits) - A * (1 << (pe_of(k, par) - 1)));
}

// The same for a word known to hold no -128 byte (the quantizer's own output:
// |x * id| stays below 127.5, so every code is in -127..127): q' = word and
// A = sum(q').
__device__ __forceinline__ void lane_consts_no_m128(uint32_t word, int k, int par, uint32_t& qp, uint32_t& ci) {
  qp = word;
  const int A = __dp4a(int(word), 0x01010101, 0);
  ci = uint32_t(int(kMagicBits) - A * (1 << (pe_of(k, par) - 1)));
}

__device__ __forceinline__ void scale_consts(float d1, int k, int par, float& dprime, float& K) {
  dprime = __fmul_rn(d1, pow2i(1 - pe_of(k, par)));
  K = -__fmul_rn(dprime, kMagic);
}

// The Q1_0 constants as the table builders take them (another format passes
// its own pair; the table's geometry is shared).
struct ConstsQ1 {
  static __device__ __forceinline__ void lane(uint32_t word, int k, int par, uint32_t& qp, uint32_t& ci) {
    lane_consts(word, k, par, qp, ci);
  }
  static __device__ __forceinline__ void lane_no_m128(uint32_t word, int k, int par, uint32_t& qp, uint32_t& ci) {
    lane_consts_no_m128(word, k, par, qp, ci);
  }
  static __device__ __forceinline__ void scale(float d1, int k, int par, float& dprime, float& K) {
    scale_consts(d1, k, par, dprime, K);
  }
};

// Table for blocks [blk0, blk0 + kcb) from a quantized activation (q int8 [n],
// d fp16 [n/32]), written at table positions tpos0 .. tpos0 + kcb - 1 of a
// table of kc blocks.  Sub-blocks past the activation's end get zero constants.
// Both builders issue the global loads of kTableBatch rounds (a round: one
// entry per thread) before using any of them, so their latencies overlap; a
// larger batch holds more registers across the call, and the caller picks the
// largest that its kernel affords without spilling.
// table_q_body is the builder itself, for kernels that inline it (loads the
// caller has in flight then stay in flight); build_table_q is the same as an
// out-of-line call.
template <int kTableBatch, class C>
__device__ __forceinline__ void table_q_body(const int8_t* __restrict__ q, const uint16_t* __restrict__ d1, int nb,
                                             int blk0, int kcb, unsigned char* table, int tid, int nthreads, int kc,
                                             int tpos0) {
  uint4* QC = reinterpret_cast<uint4*>(table) + tpos0 * 16;
  float4* DK = reinterpret_cast<float4*>(table + table_dk_offset(kc)) + tpos0 * 4;
  const int nsub = nb * 4;
  for (int base = 0; base < kcb * 16; base += kTableBatch * nthreads) {
    uint32_t wb[kTableBatch][2];
#pragma unroll
    for (int u = 0; u < kTableBatch; ++u) {
      const int t = base + u * nthreads + tid;
      const int G = blk0 * 4 + (t >> 2), w = t & 3;
#pragma unroll
      for (int par = 0; par < 2; ++par) {
        wb[u][par] = 0u;
        if (t < kcb * 16 && G < nsub)
          wb[u][par] = *reinterpret_cast<const uint32_t*>(q + int64_t(G) * kSub + 4 * (w + 4 * par));
      }
    }
#pragma unroll
    for (int u = 0; u < kTableBatch; ++u) {
      const int t = base + u * nthreads + tid;
      if (t >= kcb * 16) break;
      const int g = t >> 2, w = t & 3;
      uint32_t qp[2], ci[2];
#pragma unroll
      for (int par = 0; par < 2; ++par) C::lane(wb[u][par], g & 3, par, qp[par], ci[par]);
      QC[g * 4 + w] = make_uint4(qp[0], qp[1], ci[0], ci[1]);
    }
  }
  for (int base = 0; base < kcb * 4; base += kTableBatch * nthreads) {
    uint16_t hb[kTableBatch];
#pragma unroll
    for (int u = 0; u < kTableBatch; ++u) {
      const int g = base + u * nthreads + tid;
      const int G = blk0 * 4 + g;
      hb[u] = (g < kcb * 4 && G < nsub) ? d1[G] : uint16_t(0);
    }
#pragma unroll
    for (int u = 0; u < kTableBatch; ++u) {
      const int g = base + u * nthreads + tid;
      if (g >= kcb * 4) break;
      const float dv = __half2float(__ushort_as_half(hb[u]));
      float de, dodd, ke, ko;
      C::scale(dv, g & 3, 0, de, ke);
      C::scale(dv, g & 3, 1, dodd, ko);
      DK[g] = make_float4(de, dodd, ke, ko);
    }
  }
}

template <int kTableBatch, class C = ConstsQ1>
static __device__ __noinline__ void build_table_q(const int8_t* __restrict__ q, const uint16_t* __restrict__ d1,
                                              int nb, int blk0, int kcb, unsigned char* table, int tid,
                                              int nthreads, int kc) {
  table_q_body<kTableBatch, C>(q, d1, nb, blk0, kcb, table, tid, nthreads, kc, 0);
}

// roundf(t) (halves away from zero) as an 8-bit two's-complement code, for
// |t| < 2^22, with floating-point adds on the FMA pipe instead of conversion
// instructions.  With s = |t| + 1/2 exact, k = floor(s) = roundf(|t|) is an
// integer with k <= s; rounding toward zero is monotone and keeps k, so
// a = RZ(s) lies in [k, s] and floor(a) = k.  Between 2^23 and 2^24 floats are
// the integers, so RZ(a + 2^23) = 2^23 + k exactly and its low bits are k.
// The sign of t is then applied in two's complement.  (t = +-0 gives 0.)
__device__ __forceinline__ uint32_t round_code(float t) {
  const float a = __fadd_rz(fabsf(t), 0.5f);
  const uint32_t k = __float_as_uint(__fadd_rz(a, 8388608.0f));  // 0x4B000000 + k
  const uint32_t neg = 0u - (__float_as_uint(t) >> 31);          // all ones when t < 0
  return ((k ^ neg) - neg) & 0xffu;
}

// The four q8_0 codes of v (x * id per element, rounded as above) in one word,
// element 0 in the low byte.
__device__ __forceinline__ uint32_t quant_word(const float4& v, float id) {
  const uint32_t c0 = round_code(__fmul_rn(v.x, id)), c1 = round_code(__fmul_rn(v.y, id));
  const uint32_t c2 = round_code(__fmul_rn(v.z, id)), c3 = round_code(__fmul_rn(v.w, id));
  return c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
}

// Table for blocks [blk0, blk0 + kcb) (at table positions from tpos0, as
// above) from an f32 activation x [n], quantizing it on the way exactly as
// q8_quantize_act does (per 32 values: amax, d = amax/127, id = d ? 1/d : 0,
// q = roundf(x*id), scale fp16(d)).  One thread per (sub-block, word w): the
// lanes w and w + 4, i.e. elements 4w..4w+3 and 16+4w..16+4w+3, which fill one
// QC entry; the 4 threads of a sub-block are consecutive in a warp and share
// amax by two shuffles; thread w = 0 writes the sub-block's DK entry.  A round
// of a warp whose first thread is past the end is skipped (the whole warp
// agrees); nthreads must be a multiple of 32 and every thread of the group
// must call.  table_x_body inlined, build_table_x out of line, as for the
// quantized form.
template <int kTableBatch, class C>
__device__ __forceinline__ void table_x_body(const float* __restrict__ x, int nb, int blk0, int kcb,
                                             unsigned char* table, int tid, int nthreads, int kc, int tpos0) {
  uint4* QC = reinterpret_cast<uint4*>(table) + tpos0 * 16;
  float4* DK = reinterpret_cast<float4*>(table + table_dk_offset(kc)) + tpos0 * 4;
  const int nsub = nb * 4;
  const int total = kcb * 16;
  const int warp0 = tid & ~31;
  for (int base = 0; base < total; base += kTableBatch * nthreads) {  // same trip count for every thread
    float4 lo[kTableBatch], hi[kTableBatch];
#pragma unroll
    for (int u = 0; u < kTableBatch; ++u) {
      const int t = base + u * nthreads + tid;
      const int G = blk0 * 4 + (t >> 2), w = t & 3;
      lo[u] = hi[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < total && G < nsub) {
        const float* xs = x + int64_t(G) * kSub + 4 * w;
        lo[u] = *reinterpret_cast<const float4*>(xs);
        hi[u] = *reinterpret_cast<const float4*>(xs + 16);
      }
    }
#pragma unroll
    for (int u = 0; u < kTableBatch; ++u) {
      if (base + u * nthreads + warp0 >= total) break;  // uniform in the warp
      const int t = base + u * nthreads + tid;
      const int g = t >> 2, w = t & 3;
      const int G = blk0 * 4 + g;
      const float4 a = lo[u], b = hi[u];
      float amax = fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                         fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const float dd = __fdiv_rn(amax, 127.0f);
      const float id = (dd != 0.0f) ? __fdiv_rn(1.0f, dd) : 0.0f;
      const uint32_t wlo = quant_word(a, id), whi = quant_word(b, id);
      if (t < total) {
        const int k = g & 3;
        uint32_t qp0, ci0, qp1, ci1;
        C::lane_no_m128(wlo, k, 0, qp0, ci0);
        C::lane_no_m128(whi, k, 1, qp1, ci1);
        QC[g * 4 + w] = make_uint4(qp0, qp1, ci0, ci1);
        if (w == 0) {
          const float d1 = G < nsub ? __half2float(__float2half_rn(dd)) : 0.0f;
          float de, dodd, ke, ko;
          C::scale(d1, k, 0, de, ke);
          C::scale(d1, k, 1, dodd, ko);
          DK[g] = make_float4(de, dodd, ke, ko);
        }
      }
    }
  }
}

template <int kTableBatch, class C = ConstsQ1>
static __device__ __noinline__ void build_table_x(const float* __restrict__ x, int nb, int blk0, int kcb,
                                              unsigned char* table, int tid, int nthreads, int kc) {
  table_x_body<kTableBatch, C>(x, nb, blk0, kcb, table, tid, nthreads, kc, 0);
}

template <int I>
__device__ __forceinline__ uint32_t word_at(const uint4& v) {
  if constexpr (I == 0) return v.x;
  else if constexpr (I == 1) return v.y;
  else if constexpr (I == 2) return v.z;
  else return v.w;
}

// fp16 scale I (0..3) of a quad held as 4 halves in a uint2.
template <int I>
__device__ __forceinline__ float quad_scale(const uint2& v) {
  const uint32_t w = (I < 2) ? v.x : v.y;
  return __half2float(__ushort_as_half(uint16_t((I & 1) ? (w >> 16) : (w & 0xffffu))));
}

// Sub-block K of block BQ of a quad for R rows and one word (lanes w and
// w+4): masks each row's word to the two lanes' planes and forms the exact
// products d1*s, then ab = d1*s (K = 0) or add.rn(ab, d1*s) (K > 0) for lane
// w (abE) and lane w+4 (abO).  QCq/DKq point at the quad's first sub-block.
// The chains are scalar f32 operations: the dp4a already occupies the
// FMA-heavy pipe, and scalar fma/add can issue to either FMA pipe, where the
// paired f32x2 forms load the heavy pipe as well.
template <int R, int BQ, int K>
__device__ __forceinline__ void quad_subblock(const uint4 (&wv)[R], const uint4* QCq, const float4* DKq, int w,
                                              float (&abE)[R], float (&abO)[R]) {
  const uint4 qc = QCq[(BQ * 4 + K) * 4 + w];
  const float4 dk = DKq[BQ * 4 + K];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint32_t W = word_at<BQ>(wv[r]);
    uint32_t m0 = W & (0x01010101u << (2 * K));
    const uint32_t m1 = W & (0x01010101u << (2 * K + 1));
    if constexpr (K == 0) m0 <<= 1;  // plane 0 is used as plane 1 (byte values 0/2)
    const float pE = __fmaf_rn(dk.x, __uint_as_float(dp4a_us(m0, qc.x, qc.z)), dk.z);
    const float pO = __fmaf_rn(dk.y, __uint_as_float(dp4a_us(m1, qc.y, qc.w)), dk.w);
    if constexpr (K == 0) {
      abE[r] = pE;
      abO[r] = pO;
    } else {
      abE[r] = __fadd_rn(abE[r], pE);
      abO[r] = __fadd_rn(abO[r], pO);
    }
  }
}

// Block BQ of a quad for R rows: the four sub-blocks, then the outer
// acc = fma(d0, ab, acc) with d0 the row's block scale, per lane.
template <int R, int BQ>
__device__ __forceinline__ void quad_block(const uint4 (&wv)[R], const uint2 (&sc)[R], const uint4* QCq,
                                           const float4* DKq, int w, float (&accE)[R], float (&accO)[R]) {
  float abE[R], abO[R];
  quad_subblock<R, BQ, 0>(wv, QCq, DKq, w, abE, abO);
  quad_subblock<R, BQ, 1>(wv, QCq, DKq, w, abE, abO);
  quad_subblock<R, BQ, 2>(wv, QCq, DKq, w, abE, abO);
  quad_subblock<R, BQ, 3>(wv, QCq, DKq, w, abE, abO);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float d0 = quad_scale<BQ>(sc[r]);
    accE[r] = __fmaf_rn(d0, abE[r], accE[r]);
    accO[r] = __fmaf_rn(d0, abO[r], accO[r]);
  }
}

// A whole quad (4 blocks) for R rows: accE[r] is lane w's chain of row r,
// accO[r] lane w+4's.
template <int R>
__device__ __forceinline__ void quad_all(const uint4 (&wv)[R], const uint2 (&sc)[R], const uint4* QCq,
                                         const float4* DKq, int w, float (&accE)[R], float (&accO)[R]) {
  quad_block<R, 0>(wv, sc, QCq, DKq, w, accE, accO);
  quad_block<R, 1>(wv, sc, QCq, DKq, w, accE, accO);
  quad_block<R, 2>(wv, sc, QCq, DKq, w, accE, accO);
  quad_block<R, 3>(wv, sc, QCq, DKq, w, accE, accO);
}

// Horizontal sum of a row: thread w holds (a_w, a_w+4) and adds them; xor 2
// then gives (a0+a4)+(a2+a6) and (a1+a5)+(a3+a7), xor 1 joins the two.  All
// 32 lanes of the warp take part; the row's sum ends up in every thread of
// its group of four.
__device__ __forceinline__ float row_sum(float accE, float accO) {
  float sum = __fadd_rn(accE, accO);
  sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 2));
  return __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 1));
}

}  // namespace q1
