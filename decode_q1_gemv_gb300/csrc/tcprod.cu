// tcprod.cu -- the batched Q1_0 x q8_0 product on the tensor core: the path
// of q1_0_gemm_small for groups of 16 activation vectors.
//
// Definition (bankML "docs/modules/gpu.md", "kernels.rs -- the Q1_0 kernels",
// first and second bullets): per row, lane l and block b the chain
//   ab = d1_0*s_0;  ab = fma(d1_k, s_k, ab), k = 1..3;  acc_l = fma(d0, ab, acc_l)
// over exact integer lane sums s_k, then the fixed horizontal sum.  Each
// lane's chain is independent, so one pass over the weights serves every
// vector.
//
// Where the tensor core comes in.  Every d1_k*s_k is exact in f32 (at most 21
// significant bits), so each step of the ab chain rounds only the sum of two
// exact terms.  Write d1_k = m_k * 2^(e_k - 25) (fp16: m_k < 2^11) and
// u = 2^(e_min - 25), e_min = min_k e_k: every d1_k*s_k is an integer multiple
// of u, and so is every partial sum of the chain.  If for a lane
//   sum_k (m_k * 2^(e_k - e_min)) * sum_i |q_{k,i}|  <=  2^22,
// every partial sum is an integer multiple of u below 2^22 * u in magnitude,
// hence exactly representable in f32: no step of the chain rounds and
// ab = sum_k d1_k * s_k exactly.  With s_k = sum_i sigma_i q_i (sigma = +1 for
// a set sign bit, -1 for a clear one; the bound excludes q = -128, whose
// wrapped negation is not -q) this is a plain dot product of the lane's 16
// signs with y_j = d1_k(j) * q_j.  Each y_j (18 significant bits at most) splits
// into two f16 numbers, hi = f16(y_j) and lo = y_j - hi, both exact; two f16
// MMAs (A = the +-1 signs of 128 rows, B = hi resp. lo of 16 vectors, K = the
// lane's 16 elements) accumulate them into one f32 column.  All products are
// exact and every partial sum of that accumulation stays below 2^23 * u in
// magnitude, so the f32 accumulator holds ab exactly; then
// acc = fma(d0, ab, acc) runs on the CUDA cores as in the definition.  The
// bound depends on the activation only: a small prologue kernel checks it
// for every (block, 16-vector group) and prepares the B tiles.  Blocks where
// it fails (or where a -128 quant or a scale of 512 or more occurs) take the
// exact dp4a chain of table.cuh instead, from per-block tables the prologue
// writes in their place.
//
// Structure (one persistent CTA per SM, 29 warps, stages that run
// concurrently on different blocks):
//   warps 0-15  epilogue: warp (quarter q, word w) takes lanes w, w+4 of its
//               32 rows from tensor memory into acc = fma(d0, ab, acc), two
//               vectors an instruction (or runs the dp4a chain on a table
//               block); at the end of a tile the four words' partial sums
//               meet in shared memory for the horizontal sum.
//   warps 16-23 A builders: warp 16 + 4h + q owns rows 32q..32q+31 of the
//               128-row tile (tensor-memory lanes) and turns their sign words
//               2h and 2h + 1 into the +-1 f16 A operand of those words' four
//               lanes (tensor memory), up to two blocks ahead of the MMAs.
//   warps 24-27 MMA issuers: warp 24 + l issues the hi and lo MMAs of lanes
//               2l and 2l + 1 of every block (a warp issues its MMAs one
//               after the other, a hundred or more cycles each; separate
//               warps issue in parallel) and commits them once to the
//               block's completion barrier (D ready, A slot free).  The
//               whole warp runs the loop and one elected lane issues.
//   warp 28     producer: 1-D bulk copies of the tile's weight quads (4
//               blocks x 128 rows) and of each block's B record into rings.
// Each block's slot in every ring (A 2, D 3, B records 6, completion 6)
// follows from the block index modulo 6; the issuers walk their blocks six
// at a time, so their slots are compile-time constants.  The issuers' own
// instruction stream sets the pace, and all 29 warps share the SM's four
// schedulers and its ALU pipe: the roles' loops are unrolled, the builders'
// multiply-adds kept on the FMA pipe and the epilogue's fmas paired.
// Tensor memory: two A slots of 64 columns (8 lanes x 8 f16 pairs) and three
// D slots of 128 columns (8 lanes x 16 vectors).  Within a slot the two lanes
// of sign word w sit side by side (A: lane w at 16w, lane w+4 at 16w + 8;
// D: lane w at 32w, lane w+4 at 32w + 16), so each builder thread writes a
// word's two lanes with one tensor-memory copy.  Every waiter on an mbarrier
// passes its phases one by one, in order, and no barrier can run two phases
// ahead of a waiter (a parity wait cannot tell a phase from the one two
// before it).  Every wait is bounded; a wait that gives up raises a CTA-wide
// abort flag and the device status word, and every role winds down.
#include <algorithm>
#include <mutex>
#include <type_traits>
#include <cuda_fp16.h>

#include "table.cuh"
#include "tc.cuh"

namespace q1 {

static __device__ unsigned g_status_tc = 0u;

constexpr int kTcV = 16;                 // vectors per group (MMA N)
constexpr int kTcRows = 128;             // rows per tile (MMA M)
constexpr int kRecBytes = 8192;          // per (group, block): 16 B tiles of 512 B, or the slow tables
constexpr int kSlowBytes = kTcV * 320;   // 16 vectors' one-block dp4a tables (table.cuh, kc = 1)
constexpr int kEpiWarps = 16;            // warps 0-15
constexpr int kEpi = kEpiWarps * 32;
constexpr int kBuildWarp0 = 16, kBuildWarps = 8;
constexpr int kIssuerWarp0 = kBuildWarp0 + kBuildWarps, kIssuers = 4;
constexpr int kBuildWords = 16 / kBuildWarps;  // sign words a builder warp turns into A, for its 32 rows
constexpr int kIssuerLanes = 8 / kIssuers;     // lanes whose MMAs an issuer warp issues
static_assert(kBuildWarps % 4 == 0 && 16 % kBuildWarps == 0 && 8 % kIssuers == 0, "role split");
constexpr int kProducerWarp = kIssuerWarp0 + kIssuers;
constexpr int kTcThreads = 29 * 32;
constexpr int kASlots = 2, kDSlots = 3;
constexpr int kMSlots = 6;  // MMA-completion barriers: block i on i % 6, a multiple of both slot counts
constexpr int kWStages = 4;
constexpr int kBStages = 6;
static_assert(kBStages == kMSlots && kMSlots == 2 * kDSlots && kMSlots == 3 * kASlots,
              "one position (i % 6, (i / 6) & 1) gives block i's slot in every per-block ring");
constexpr int kWStageBytes = 4 * 2048 + 4 * 256;   // one quad of the tile's 4 panels: bits + scales
constexpr int kOffW = 0;
constexpr int kOffB = kOffW + kWStages * kWStageBytes;
constexpr int kOffPart = kOffB + kBStages * kRecBytes;
constexpr int kPartBytes = 4 * kTcV * kTcRows * 4;
constexpr int kOffBars = kOffPart + kPartBytes;
// barriers: wfull, wempty, bfull, bempty, afull, mdone, dempty, partfull, partfree, drain
constexpr int kBarWFull = 0, kBarWEmpty = kBarWFull + kWStages, kBarBFull = kBarWEmpty + kWStages,
              kBarBEmpty = kBarBFull + kBStages, kBarAFull = kBarBEmpty + kBStages, kBarMDone = kBarAFull + kASlots,
              kBarDEmpty = kBarMDone + kMSlots,
              kBarPartFull = kBarDEmpty + kDSlots, kBarPartFree = kBarPartFull + 1, kBarDrain = kBarPartFree + 1,
              kNumBars = kBarDrain + kIssuers;
constexpr int kOffFlag = kOffBars + kNumBars * 8;
constexpr int kOffMisc = kOffFlag + kBStages * 4;
constexpr int kTcSmem = kOffMisc + 16;
static_assert(kOffB % 1024 == 0 && kOffPart % 16 == 0, "shared-memory alignment");
static_assert(kTcSmem <= 227 * 1024, "shared-memory budget");
static_assert(kTcSmem > 114 * 1024, "one CTA per SM: the kernel takes all 512 tensor-memory columns");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD = 64 * kASlots;  // A slot a at columns 64 a, D slot d at kColD + 128 d
constexpr int kMaxWaitNs = 2000000000;

struct TcArgs {
  const uint8_t* bits;     // packed sign words
  const uint8_t* scales;   // packed fp16 block scales
  const uint8_t* flags;    // [groups][nb]: 1 = the block takes the tensor-core path
  const uint8_t* recs;     // [groups][nb][kRecBytes]
  float* out;              // [nvec][rows]
  int rows, nb, nbp, nvec, groups, units;
};

// ------------------------------------------------------------- prologue --
// One CTA per (block, group): thread (vector v, lane l).  Decides whether the
// block takes the tensor-core path for the group's 16 vectors (the bound in
// the file header, for every vector and lane) and writes the block's record:
// the B tiles, or the dp4a tables.  Columns past nvec repeat the last vector;
// their outputs are never stored.
//   B tile (lane l, hi = 0 / lo = 1) at byte (2l + part) * 512 of the record:
//   element (K index kappa, vector v) at (v/8)*256 + (kappa/8)*128 +
//   (v%8)*16 + (kappa%8)*2, the no-swizzle K-major layout of smem_desc with
//   LBO 128 and SBO 256.  K index kappa = 4k + pos(i) holds element
//   32k + 4l + i of the block, pos = (0, 2, 1, 3): the order in which the row
//   workers lay out the signs (two f16 per 32-bit column: elements 0 and 2,
//   then 1 and 3, of each sub-block).
__global__ void __launch_bounds__(128) k_tc_prep(const int8_t* __restrict__ q, const uint16_t* __restrict__ d,
                                                 int64_t n, int nb, int nvec, uint8_t* __restrict__ flags,
                                                 uint8_t* __restrict__ recs) {
  const int b = blockIdx.x, g = blockIdx.y;
  const int t = threadIdx.x, v = t >> 3, l = t & 7;
  const int vv = min(g * kTcV + v, nvec - 1);
  // q and d may be written by the preceding kernel.  Dependents are released
  // only after this wait, so the product kernel's early weight loads overlap
  // this kernel alone.
  pdl_wait();
  pdl_launch_dependents();
  const int8_t* qv = q + int64_t(vv) * n + int64_t(b) * kBlock;
  const uint16_t* dv = d + int64_t(vv) * (n / kSub) + int64_t(b) * 4;
  uint32_t qw[4];
  uint16_t dh[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    qw[k] = *reinterpret_cast<const uint32_t*>(qv + kSub * k + 4 * l);
    dh[k] = dv[k];
  }
  bool ok = true;
  uint32_t m[4], S[4];
  int e[4];
  int emin = 31;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int x = int(int8_t(qw[k] >> (8 * i)));
      ok = ok && x != -128;
      s += uint32_t(x < 0 ? -x : x);
    }
    S[k] = s;
    const int E = (dh[k] >> 10) & 31;
    ok = ok && E <= 23;                  // |d1| < 512: |y| < 65024 stays a finite f16
    m[k] = E ? (1024u | (dh[k] & 1023u)) : (dh[k] & 1023u);
    e[k] = E ? E : 1;
    emin = min(emin, e[k]);
  }
  uint64_t T = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (ok) T += (uint64_t(m[k]) << (e[k] - emin)) * S[k];   // e[k] - emin <= 22 when ok
  ok = ok && T <= (uint64_t(1) << 22);
  const int fast = __syncthreads_and(ok ? 1 : 0);
  uint8_t* rec = recs + (int64_t(g) * nb + b) * kRecBytes;
  if (t == 0) flags[int64_t(g) * nb + b] = uint8_t(fast);
  if (fast) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float d1 = __half2float(__ushort_as_half(dh[k]));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float y = __fmul_rn(d1, float(int(int8_t(qw[k] >> (8 * i)))));  // exact
        const __half hi = __float2half_rn(y);
        const __half lo = __float2half_rn(__fsub_rn(y, __half2float(hi)));     // exact
        const int kappa = 4 * k + ((i == 1) ? 2 : (i == 2) ? 1 : i);
        const int off = (v >> 3) * 256 + (kappa >> 3) * 128 + (v & 7) * 16 + (kappa & 7) * 2;
        *reinterpret_cast<__half*>(rec + (2 * l) * 512 + off) = hi;
        *reinterpret_cast<__half*>(rec + (2 * l + 1) * 512 + off) = lo;
      }
    }
  } else {
    table_q_body<1, ConstsQ1>(q + int64_t(vv) * n, d + int64_t(vv) * (n / kSub), nb, b, 1, rec + v * 320, l, 8,
                              1, 0);
  }
}

// ---------------------------------------------------------- main kernel --
// try_wait with a suspend-time hint: the thread sleeps in the barrier unit
// until the phase completes or about `ns` nanoseconds pass, issuing nothing
// meanwhile.
__device__ __forceinline__ bool mbar_try_suspend(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return done != 0;
}

// Bounded wait with a CTA-wide abort flag: false when the flag is up or after
// about two seconds (then it raises the flag).  Each round parks the thread in
// the barrier (up to 20 us): polling threads would otherwise take the issue
// slots the other roles need, and a sleep between polls would overshoot the
// phase's completion.
static __device__ __noinline__ bool tc_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_suspend(bar, parity, 20000u)) return true;
    if ((i & 7) == 0) {  // the flag and the clock every eighth round: fewer instructions a round
      if (*abort_flag) return false;
      if (globaltimer() - t0 > uint64_t(kMaxWaitNs)) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try(bar, parity)) return true;
  return tc_wait_slow(bar, parity, abort_flag);
}
// Every lane of the warp waits (each then holds the barrier's acquire); the
// warp goes on when all have seen the phase complete, and gives up with them.
// In the common case the phase is already complete: one poll and one vote.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  bool done = mbar_try(bar, parity);
  if (!done) done = tc_wait_slow(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, done);
}
// Whether the phases with the given parities of three barriers have all
// completed, tested side by side without waiting: each test is a round trip
// to the barrier unit of about a hundred cycles, which an MMA issuer would
// otherwise pay three times a block.
__device__ __forceinline__ bool mbar_test3(uint32_t b0, uint32_t p0, uint32_t b1, uint32_t p1, uint32_t b2,
                                           uint32_t p2) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred a, b, c;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 a, [%1], %2;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 b, [%3], %4;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 c, [%5], %6;\n\t"
      "and.pred a, a, b;\n\t"
      "and.pred a, a, c;\n\t"
      "selp.u32 %0, 1, 0, a; }"
      : "=r"(done)
      : "r"(b0), "r"(p0), "r"(b1), "r"(p1), "r"(b2), "r"(p2)
      : "memory");
  return done != 0;
}
// Block i's slot and phase in the per-block rings, from m = i % 6 and
// ph = (i / 6) & 1 (the MMA-completion ring and the B ring are both six
// long): the D ring (three) and the A ring (two) follow.
__device__ __forceinline__ int d_slot(int m) { return m >= 3 ? m - 3 : m; }
__device__ __forceinline__ uint32_t d_phase(int m) { return m >= 3 ? 1u : 0u; }
__device__ __forceinline__ int a_slot(int m) { return m & 1; }
__device__ __forceinline__ uint32_t a_phase(int m, uint32_t ph) { return ph ^ uint32_t((m >> 1) & 1); }
// Whether the phases with the given parities of two barriers have both
// completed (tested side by side, without waiting).
__device__ __forceinline__ bool mbar_test2(uint32_t b0, uint32_t p0, uint32_t b1, uint32_t p1) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred a, b;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 a, [%1], %2;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 b, [%3], %4;\n\t"
      "and.pred a, a, b;\n\t"
      "selp.u32 %0, 1, 0, a; }"
      : "=r"(done)
      : "r"(b0), "r"(p0), "r"(b1), "r"(p1)
      : "memory");
  return done != 0;
}
// Slot index and phase bit of a ring of N, advanced one position.
template <int N>
__device__ __forceinline__ void ring_next(int& slot, uint32_t& phase) {
  if (++slot == N) {
    slot = 0;
    phase ^= 1u;
  }
}

// Integer multiply-add on the FMA pipe (the ALU pipe carries the masks).
__device__ __forceinline__ uint32_t imad(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The negated signs -sigma (f16: -1 for a set sign bit, +1 for a clear one)
// of lane w (even planes, columns 0-7 of av) and lane w + 4 (odd planes,
// columns 8-15) of one block from its sign word: within a lane, column 2k
// holds elements 0 and 2 of sub-block k, column 2k + 1 elements 1 and 3 (low
// half first).  A sign bit masked out and multiplied onto bit 15 / 31 of
// f16 +1.0 (0x3C00) flips that half's sign: one mask and one multiply-add per
// column.  The accumulator then holds -ab, which the epilogue multiplies by
// -d0 (an exact negation: fma(-d0, -ab, acc) = fma(d0, ab, acc)).
__device__ __forceinline__ void signs_to_f16(uint32_t W, uint32_t (&av)[16]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int par = 0; par < 2; ++par) {
      const int pl = 2 * k + par;
      // Each multiplier carries a second term that moves both masked bits
      // past bit 31, where they vanish: not a power of two, it stays an
      // integer multiply-add on the FMA pipe instead of a shift-add on the
      // ALU pipe, which the masks and the control code already load.
      av[8 * par + 2 * k] =
          imad(W & (0x00010001u << pl), (1u << (15 - pl)) + (pl > 0 ? 1u << ((32 - pl) & 31) : 0u), 0x3C003C00u);
      av[8 * par + 2 * k + 1] = imad(W & (0x01000100u << pl), (1u << (7 - pl)) + (1u << (24 - pl)), 0x3C003C00u);
    }
  }
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int bq) {
  return bq == 0 ? v.x : bq == 1 ? v.y : bq == 2 ? v.z : v.w;
}
__device__ __forceinline__ uint32_t scale_of(const uint2& v, int bq) {
  const uint32_t x = (bq < 2) ? v.x : v.y;
  return (bq & 1) ? (x >> 16) : (x & 0xffffu);
}

__global__ void __launch_bounds__(kTcThreads, 1) k_q1_tc(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  int* bflag = reinterpret_cast<int*>(smem + kOffFlag);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(bar(kBarWFull + s), 1);
      mbar_init(bar(kBarWEmpty + s), 32 * (kEpiWarps + kBuildWarps));
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(bar(kBarBFull + s), 1);
      mbar_init(bar(kBarBEmpty + s), 32 * kEpiWarps);
    }
    for (int s = 0; s < kASlots; ++s) mbar_init(bar(kBarAFull + s), 32 * kBuildWarps);
    for (int s = 0; s < kMSlots; ++s) mbar_init(bar(kBarMDone + s), kIssuers);
    for (int s = 0; s < kDSlots; ++s) mbar_init(bar(kBarDEmpty + s), 32 * kEpiWarps);
    // Barriers the row workers release are arrived on by every lane of their
    // warps (each lane after its own accesses), the others by one thread.
    mbar_init(bar(kBarPartFull), 32 * kEpiWarps);
    mbar_init(bar(kBarPartFree), 32 * kEpiWarps);
    for (int i = 0; i < kIssuers; ++i) mbar_init(bar(kBarDrain + i), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int nq = (a.nb + 3) / 4;  // quads that hold real blocks

  if (warp == kProducerWarp) {
    // ------------------------------------------------------- producer --
    if (lane == 0) {
      auto copy_quad = [&](int s, int64_t p0, int qd) {
        const uint32_t wf = bar(kBarWFull + s);
        mbar_arrive_expect_tx(wf, uint32_t(kWStageBytes));
        const uint32_t dst = smem_addr(smem + kOffW + s * kWStageBytes);
        bulk_g2s(dst, a.bits + quad_bits_offset(p0, qd, a.nbp), 4 * 2048, wf);
        bulk_g2s(dst + 4 * 2048, a.scales + quad_scales_offset(p0, qd, a.nbp), 4 * 256, wf);
      };
      // The weights do not depend on the prologue kernel: the first unit's
      // first quads go out before waiting for it (the builders can start on
      // them); the records and their flags are the prologue's output.
      const int pre = blockIdx.x < unsigned(a.units) ? min(nq, kWStages) : 0;
      for (int qd = 0; qd < pre; ++qd)
        copy_quad(qd, int64_t(int(blockIdx.x) / a.groups) * (kTcRows / kPanel), qd);
      pdl_wait();
      int wq = 0, it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        const int t = u / a.groups, g = u % a.groups;
        const int64_t p0 = int64_t(t) * (kTcRows / kPanel);
        for (int qd = 0; qd < nq && ok; ++qd, ++wq) {
          const int s = wq % kWStages;
          if (wq >= pre) {
            if (wq >= kWStages && !tc_wait(bar(kBarWEmpty + s), uint32_t(wq / kWStages - 1) & 1u, abort_flag)) {
              ok = false;
              break;
            }
            copy_quad(s, p0, qd);
          }
          for (int bq = 0; bq < 4 && qd * 4 + bq < a.nb; ++bq, ++it) {
            const int b = qd * 4 + bq, s2 = it % kBStages;
            if (it >= kBStages && !tc_wait(bar(kBarBEmpty + s2), uint32_t(it / kBStages - 1) & 1u, abort_flag)) {
              ok = false;
              break;
            }
            const int fast = a.flags[int64_t(g) * a.nb + b];
            bflag[s2] = fast;
            const uint32_t bytes = fast ? uint32_t(kRecBytes) : uint32_t(kSlowBytes);
            const uint32_t bf = bar(kBarBFull + s2);
            mbar_arrive_expect_tx(bf, bytes);
            bulk_g2s(smem_addr(smem + kOffB + s2 * kRecBytes), a.recs + (int64_t(g) * a.nb + b) * kRecBytes, bytes,
                     bf);
          }
        }
      }
      // The CTA's shared memory must outlive every copy issued into it.
      for (int k = max(0, wq - kWStages); k < wq; ++k)
        mbar_wait(bar(kBarWFull + k % kWStages), uint32_t(k / kWStages) & 1u, 100000000ull);
      for (int k = max(0, it - kBStages); k < it; ++k)
        mbar_wait(bar(kBarBFull + k % kBStages), uint32_t(k / kBStages) & 1u, 100000000ull);
    }
  } else if (warp >= kIssuerWarp0) {
    // ---------------------------------------------------------- issuers --
    // Warp kIssuerWarp0 + l: lanes 2l and 2l + 1 of every block.  The whole
    // warp runs the loop and one elected lane issues: the slot and address
    // arithmetic stays warp-uniform.
    const int l = warp - kIssuerWarp0;
    const uint32_t idesc = idesc_f16(kTcRows, kTcV);
    // Loop-invariant parts of the operands.  A descriptor's start address is
    // its low 14 bits in 16-byte units, and every B tile lies well inside that
    // range, so a tile's descriptor is the region's plus its offset / 16.
    const uint64_t bdesc0 = smem_desc(smem_addr(smem + kOffB), 128, 256);
    uint32_t dlane[kIssuerLanes], alane[kIssuerLanes];
    uint64_t blane[kIssuerLanes];
#pragma unroll
    for (int j = 0; j < kIssuerLanes; ++j) {
      const int ll = kIssuerLanes * l + j;
      dlane[j] = tbase + kColD + 32u * uint32_t(ll & 3) + 16u * uint32_t(ll >> 2);
      alane[j] = tbase + 16u * uint32_t(ll & 3) + 8u * uint32_t(ll >> 2);
      blane[j] = bdesc0 + uint64_t((2 * ll * 512) >> 4);
    }
    // The CTA's blocks in order, six at a time: a block's slot in every ring
    // is its index modulo 6, a compile-time constant in the unrolled loop, and
    // only the phase bit of the six-block round varies.
    const int total = (a.units - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x) * a.nb;
    uint32_t mph = 0;
    bool ok = true;
    int it0 = 0;
    // Block m of a round (phase bit mph): false when a wait gave up.
    auto issue = [&](auto mc) -> bool {
      constexpr int m = decltype(mc)::value;
      constexpr int asl = m & 1, dsl = m >= 3 ? m - 3 : m, s2 = m;
      const uint32_t aph = mph ^ uint32_t((m >> 1) & 1), dph = m >= 3 ? 1u : 0u, bph = mph;
      // The A slot is built, the D slot is free (a fresh barrier counts its
      // phase of parity 1 as complete: the first kDSlots blocks pass) and the
      // B record has landed.
      const bool ready =
          mbar_test3(bar(kBarAFull + asl), aph, bar(kBarDEmpty + dsl), dph ^ 1u, bar(kBarBFull + s2), bph);
      if (!__all_sync(0xffffffffu, ready) &&
          (!warp_wait(bar(kBarAFull + asl), aph, abort_flag) ||
           !warp_wait(bar(kBarDEmpty + dsl), dph ^ 1u, abort_flag) ||
           !warp_wait(bar(kBarBFull + s2), bph, abort_flag)))
        return false;
      tc_fence_after();
      if (bflag[s2]) {
        constexpr uint32_t doff = 128u * dsl, aoff = 64u * asl;
        constexpr uint64_t boff = uint64_t(s2 * (kRecBytes >> 4));
#pragma unroll
        for (int j = 0; j < kIssuerLanes; ++j) {  // this issuer's lanes: hi tile, then lo tile 512 B on
          mma_f16_ts_elect(dlane[j] + doff, alane[j] + aoff, blane[j] + boff, idesc, 0u);
          mma_f16_ts_elect(dlane[j] + doff, alane[j] + aoff, blane[j] + boff + (512 >> 4), idesc, 1u);
        }
      }
      mma_commit_elect(bar(kBarMDone + m));  // D ready and A slot free
      return true;
    };
    // Whole rounds without bounds checks, then the last partial round.
    using I0 = std::integral_constant<int, 0>;
    using I1 = std::integral_constant<int, 1>;
    using I2 = std::integral_constant<int, 2>;
    using I3 = std::integral_constant<int, 3>;
    using I4 = std::integral_constant<int, 4>;
    using I5 = std::integral_constant<int, 5>;
    const int whole = total - total % kMSlots;
    for (; it0 < whole && ok; it0 += kMSlots, mph ^= 1u)
      ok = issue(I0{}) && issue(I1{}) && issue(I2{}) && issue(I3{}) && issue(I4{}) && issue(I5{});
    if (ok && it0 < total) {
      const int rest = total - it0;  // 1 to 5 blocks
      ok = issue(I0{});
      if (ok && rest > 1) ok = issue(I1{});
      if (ok && rest > 2) ok = issue(I2{});
      if (ok && rest > 3) ok = issue(I3{});
      if (ok && rest > 4) ok = issue(I4{});
    }
    // After an abort, this issuer's MMAs may still be running: a commit to its
    // own drain barrier arrives once they are all through (at once if there
    // are none); wait for it (bounded) before the tensor memory is released.
    if (!ok) {
      mma_commit_elect(bar(kBarDrain + l));
      if (lane == 0) mbar_wait(bar(kBarDrain + l), 0u, 100000000ull);
    }
    __syncwarp();
  } else if (warp >= kBuildWarp0) {
    // ------------------------------------------------------- A builders --
    const int quarter = warp & 3, grp = (warp - kBuildWarp0) >> 2;  // words kBuildWords grp ... + kBuildWords - 1
    const uint32_t lrow = tbase + (uint32_t(quarter * 32) << 16);
    int it = 0, ws = 0, asl = 0, msl = 0;  // msl, mph: MMA-completion barrier of block it - kASlots
    uint32_t wph = 0, aph = 0, mph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
      for (int b0 = 0; b0 < a.nb; b0 += 4) {
        // A weight quad: this warp's two sign words (each holds the word of
        // the quad's four blocks) for its 32 rows.
        if (!warp_wait(bar(kBarWFull + ws), wph, abort_flag)) {
          ok = false;
          break;
        }
        const unsigned char* st = smem + kOffW + ws * kWStageBytes + quarter * 2048 + lane * 64;
        uint4 wq[kBuildWords];
#pragma unroll
        for (int jj = 0; jj < kBuildWords; ++jj)
          wq[jj] = *reinterpret_cast<const uint4*>(st + (kBuildWords * grp + jj) * 16);
        mbar_arrive(bar(kBarWEmpty + ws));
        ring_next<kWStages>(ws, wph);
#pragma unroll
        for (int bq = 0; bq < 4; ++bq) {  // the quad's blocks, unrolled: word and slot arithmetic fold
          if (b0 + bq >= a.nb) break;
          // The slot's previous block must be through its MMAs.
          if (it >= kASlots) {
            if (!warp_wait(bar(kBarMDone + msl), mph, abort_flag)) {
              ok = false;
              break;
            }
            ring_next<kMSlots>(msl, mph);
          }
          tc_fence_after();
#pragma unroll
          for (int jj = 0; jj < kBuildWords; ++jj) {
            uint32_t av[16];
            signs_to_f16(word_of(wq[jj], bq), av);
            tmem_st16(lrow + 64u * uint32_t(asl) + 16u * uint32_t(kBuildWords * grp + jj), av);
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(kBarAFull + asl));
          ring_next<kASlots>(asl, aph);
          ++it;
        }
        if (!ok) break;
      }
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int quarter = warp & 3, w = warp >> 2;
    const int rt = quarter * 32 + lane;               // row within the tile = tensor-memory lane
    const uint32_t lrow = tbase + (uint32_t(quarter * 32) << 16);
    float* part = reinterpret_cast<float*>(smem + kOffPart);  // [word][vector][row]
    int ws = 0, msl = 0, units_done = 0;
    uint32_t wph = 0, mph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x, ++units_done) {
      if (u + int(gridDim.x) >= a.units && threadIdx.x == 0) pdl_launch_dependents();
      const int t = u / a.groups, g = u % a.groups;
      // Vectors 2i and 2i + 1 side by side: the paired fma (two single
      // roundings in one instruction) halves the epilogue's issue slots.
      float2 accE[kTcV / 2], accO[kTcV / 2];
#pragma unroll
      for (int i = 0; i < kTcV / 2; ++i) accE[i] = accO[i] = make_float2(0.0f, 0.0f);
      for (int b0 = 0; b0 < a.nb && ok; b0 += 4) {
        // A weight quad: the row's word w and block scales of four blocks.
        if (!warp_wait(bar(kBarWFull + ws), wph, abort_flag)) {
          ok = false;
          break;
        }
        const unsigned char* st = smem + kOffW + ws * kWStageBytes;
        const uint4 wv = *reinterpret_cast<const uint4*>(st + quarter * 2048 + (lane * 16 + w * 4) * 4);
        const uint2 sc = *reinterpret_cast<const uint2*>(st + 4 * 2048 + quarter * 256 + lane * 8);
        mbar_arrive(bar(kBarWEmpty + ws));
        ring_next<kWStages>(ws, wph);
#pragma unroll
        for (int bq = 0; bq < 4; ++bq) {  // the quad's blocks, unrolled
          if (b0 + bq >= a.nb) break;
          const uint32_t W = word_of(wv, bq), D0 = scale_of(sc, bq);
          const int dsl = d_slot(msl), s2 = msl;
          // The block's MMAs are done and its B record has landed.
          const bool ready = mbar_test2(bar(kBarMDone + msl), mph, bar(kBarBFull + s2), mph);
          if (!__all_sync(0xffffffffu, ready) &&
              (!warp_wait(bar(kBarMDone + msl), mph, abort_flag) || !warp_wait(bar(kBarBFull + s2), mph, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (bflag[s2]) {
            // The accumulator holds -ab (signs_to_f16).
            const float d0 = -__half2float(__ushort_as_half(uint16_t(D0)));
            uint32_t dv[16];
            tmem_ld16(lrow + kColD + 128u * uint32_t(dsl) + 32u * uint32_t(w), dv);
            tmem_wait_ld16(dv);
#pragma unroll
            for (int i = 0; i < kTcV / 2; ++i)
              accE[i] = __ffma2_rn(make_float2(d0, d0),
                                   make_float2(__uint_as_float(dv[2 * i]), __uint_as_float(dv[2 * i + 1])), accE[i]);
            tmem_ld16(lrow + kColD + 128u * uint32_t(dsl) + 32u * uint32_t(w) + 16u, dv);
            tmem_wait_ld16(dv);
            tc_fence_before();
            mbar_arrive(bar(kBarDEmpty + dsl));   // D slot free for the next block
#pragma unroll
            for (int i = 0; i < kTcV / 2; ++i)
              accO[i] = __ffma2_rn(make_float2(d0, d0),
                                   make_float2(__uint_as_float(dv[2 * i]), __uint_as_float(dv[2 * i + 1])), accO[i]);
          } else {
            tc_fence_before();
            mbar_arrive(bar(kBarDEmpty + dsl));
            const unsigned char* tabs = smem + kOffB + s2 * kRecBytes;
            const uint4 wv1[1] = {make_uint4(W, 0u, 0u, 0u)};
            const uint2 sc1[1] = {make_uint2(D0, 0u)};
#pragma unroll
            for (int v = 0; v < kTcV; ++v) {
              float aE[1] = {(v & 1) ? accE[v / 2].y : accE[v / 2].x}, aO[1] = {(v & 1) ? accO[v / 2].y : accO[v / 2].x};
              quad_block<1, 0>(wv1, sc1, reinterpret_cast<const uint4*>(tabs + v * 320),
                               reinterpret_cast<const float4*>(tabs + v * 320 + 256), w, aE, aO);
              if (v & 1) {
                accE[v / 2].y = aE[0];
                accO[v / 2].y = aO[0];
              } else {
                accE[v / 2].x = aE[0];
                accO[v / 2].x = aO[0];
              }
            }
          }
          mbar_arrive(bar(kBarBEmpty + s2));
          ring_next<kMSlots>(msl, mph);
        }
      }
      if (!ok) break;
      // Horizontal sum: word w holds (a_w, a_w+4); the four words meet in
      // shared memory: ((a0+a4) + (a2+a6)) + ((a1+a5) + (a3+a7)).
      if (units_done > 0 && !warp_wait(bar(kBarPartFree), uint32_t(units_done - 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int v = 0; v < kTcV; ++v)
        part[(w * kTcV + v) * kTcRows + rt] = (v & 1) ? __fadd_rn(accE[v / 2].y, accO[v / 2].y)
                                                      : __fadd_rn(accE[v / 2].x, accO[v / 2].x);
      mbar_arrive(bar(kBarPartFull));
      if (!warp_wait(bar(kBarPartFull), uint32_t(units_done) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      for (int idx = threadIdx.x; idx < kTcV * kTcRows; idx += kEpi) {
        const int v = idx / kTcRows, r = idx % kTcRows;
        const float s = __fadd_rn(__fadd_rn(part[(0 * kTcV + v) * kTcRows + r], part[(2 * kTcV + v) * kTcRows + r]),
                                  __fadd_rn(part[(1 * kTcV + v) * kTcRows + r], part[(3 * kTcV + v) * kTcRows + r]));
        const int64_t row = int64_t(t) * kTcRows + r;
        const int vv = g * kTcV + v;
        if (row < a.rows && vv < a.nvec) a.out[int64_t(vv) * a.rows + row] = s;
      }
      mbar_arrive(bar(kBarPartFree));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_free(tbase, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_status_tc, kStatusWaitTimeout);
}

// ---------------------------------------------------------------- host ----
int status_word_tc(unsigned* v, int clear) {
  if (int e = cuda_status(cudaMemcpyFromSymbol(v, g_status_tc, sizeof *v), "q1_device_status")) return e;
  if (clear && *v) {
    const unsigned zero = 0;
    return cuda_status(cudaMemcpyToSymbol(g_status_tc, &zero, sizeof zero), "q1_device_status");
  }
  return Q1_OK;
}

// Scratch bytes of the tensor-core path: the flags, then the records.
int64_t tc_scratch_bytes(int64_t n, int64_t nvec) {
  const int64_t nb = n / kBlock, groups = (nvec + kTcV - 1) / kTcV;
  return (groups * nb + 255) / 256 * 256 + groups * nb * kRecBytes;
}

int launch_tc(const void* packed, int64_t rows, int64_t n, int64_t nvec, const int8_t* q, const uint16_t* d,
              float* out, uint8_t* scratch, cudaStream_t s, const char* who) {
  const Layout L = layout_of(rows, n);
  const int groups = int((nvec + kTcV - 1) / kTcV);
  const int64_t nb = L.nb;
  uint8_t* flags = scratch;
  uint8_t* recs = scratch + (groups * nb + 255) / 256 * 256;

  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!attr_done[dev]) {
    if (int e = cuda_status(cudaFuncSetAttribute(k_q1_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem),
                            "cudaFuncSetAttribute"))
      return e;
    attr_done[dev] = 1;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;

  cudaLaunchConfig_t cp = {};
  cp.gridDim = dim3(unsigned(nb), unsigned(groups));
  cp.blockDim = dim3(128);
  cp.stream = s;
  cp.attrs = attr;
  cp.numAttrs = 1;
  if (int e = cuda_status(cudaLaunchKernelEx(&cp, k_tc_prep, q, d, n, int(nb), int(nvec), flags, recs), who))
    return e;

  TcArgs a = {};
  a.bits = static_cast<const uint8_t*>(packed);
  a.scales = a.bits + L.bits_bytes;
  a.flags = flags;
  a.recs = recs;
  a.out = out;
  a.rows = int(rows);
  a.nb = int(nb);
  a.nbp = int(L.nbp);
  a.nvec = int(nvec);
  a.groups = groups;
  const int64_t tiles = (rows + kTcRows - 1) / kTcRows;
  a.units = int(tiles * groups);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(std::min<int64_t>(a.units, num_sms())));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = size_t(kTcSmem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, k_q1_tc, a), who);
}

}  // namespace q1

// ------------------------------------------- allocation-free batched call --
// q1_0_gemm_small_noalloc: the tensor-core batched product with its scratch
// (the prologue's flags and B records) in one array that lives in this
// library's own device memory from load to exit, for callers that cannot
// allocate device memory while they run (see q1gemv.h).
namespace q1 {

constexpr int64_t kNoAllocScratchBytes = int64_t(8) << 20;  // 8 MiB on every device that loads the library
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array on the current device.  The host-side name of a
// __device__ array is only a handle: the address a kernel may use comes from
// cudaGetSymbolAddress with that device current, looked up once per device.
static int noalloc_scratch(uint8_t** out) {
  static std::mutex lock;
  static uint8_t* addr[64] = {};
  int dev = 0;
  if (int e = cuda_status(cudaGetDevice(&dev), "q1_0_gemm_small_noalloc")) return e;
  if (dev < 0 || dev >= 64) return fail(Q1_ERR_ARG, "q1_0_gemm_small_noalloc: device %d outside 0..63", dev);
  std::lock_guard<std::mutex> g(lock);
  if (!addr[dev]) {
    void* p = nullptr;
    if (int e = cuda_status(cudaGetSymbolAddress(&p, g_noalloc_scratch),
                            "q1_0_gemm_small_noalloc: cudaGetSymbolAddress"))
      return e;
    addr[dev] = static_cast<uint8_t*>(p);
  }
  *out = addr[dev];
  return Q1_OK;
}

}  // namespace q1

extern "C" int q1_0_gemm_small_noalloc(const void* packed, int64_t rows, int64_t n, int64_t nvec, const int8_t* q,
                                       const uint16_t* d, float* out, void* stream) {
  using namespace q1;
  const char* who = "q1_0_gemm_small_noalloc";
  if (rows < 1 || rows > (int64_t(1) << 26) || n < 128 || n > (int64_t(1) << 24) || n % 128)
    return fail(Q1_ERR_ARG, "%s: bad shape rows=%lld n=%lld", who, (long long)rows, (long long)n);
  if (nvec < 1 || nvec > 64) return fail(Q1_ERR_ARG, "%s: nvec=%lld outside 1..64", who, (long long)nvec);
  if (!packed || !q || !d || !out) return fail(Q1_ERR_ARG, "%s: null pointer", who);
  if (reinterpret_cast<uintptr_t>(packed) % 16 || reinterpret_cast<uintptr_t>(q) % 16 ||
      reinterpret_cast<uintptr_t>(d) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
    return fail(Q1_ERR_ARG, "%s: buffers must be 16-byte aligned", who);
  const int64_t need = tc_scratch_bytes(n, nvec);
  if (need > kNoAllocScratchBytes)
    return fail(Q1_ERR_ARG,
                "%s: n=%lld with %lld vectors needs %lld bytes of scratch; the fixed scratch holds %lld "
                "(8 KB per 128 weights of n per group of 16 vectors)",
                who, (long long)n, (long long)nvec, (long long)need, (long long)kNoAllocScratchBytes);
  uint8_t* scratch = nullptr;
  if (int e = noalloc_scratch(&scratch)) return e;
  // Nothing in the scratch needs to start at zero: the prologue writes every
  // flag and every record byte the product kernel reads before it reads them.
  return launch_tc(packed, rows, n, nvec, q, d, out, scratch, static_cast<cudaStream_t>(stream), who);
}
