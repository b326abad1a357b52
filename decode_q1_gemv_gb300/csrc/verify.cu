// verify.cu -- q1_0_verify: the on-card self-check.  Runs every kernel of the
// library on seeded inputs and compares each output bit for bit with a
// host-side reference compiled into the library (an independent plain C++
// restatement of the definition; it never produces results for callers).
//
// Mirrors bankML "docs/modules/gpu.md", "How it is verified": random weights
// and activations including -128 quants, plus a layer-shaped regime with
// per-block scales that make products inexact in f32; one line per kernel and
// shape, or the first differing row.  The Q2_0 (ternary) product is checked
// the same way (the pages list it for --verify among the next steps).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "q2.cuh"

namespace q1 {
namespace {

// --------------------------------------------------------- host reference --
float h_half(uint16_t h) {
  const int e = (h >> 10) & 0x1f, m = h & 0x3ff;
  float v;
  if (e == 0x1f) v = m ? NAN : INFINITY;
  else if (e == 0) v = std::ldexp(float(m), -24);
  else v = std::ldexp(float(m + 1024), e - 25);
  return (h & 0x8000) ? -v : v;
}

float h_row(const uint8_t* row, int64_t nb, const int8_t* q, const uint16_t* d) {
  float a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int64_t b = 0; b < nb; ++b) {
    const uint8_t* blk = row + b * kBlockBytes;
    const float d0 = h_half(uint16_t(blk[0] | (blk[1] << 8)));
    for (int l = 0; l < 8; ++l) {
      float ab = 0.0f;
      for (int k = 0; k < 4; ++k) {
        int s = 0;
        for (int i = 0; i < 4; ++i) {
          const int j = 32 * k + 4 * l + i;
          const int qq = q[b * kBlock + j];
          const bool plus = (blk[2 + j / 8] >> (j % 8)) & 1;
          s += plus ? qq : (qq == -128 ? -128 : -qq);
        }
        const float d1 = h_half(d[b * 4 + k]);
        ab = (k == 0) ? d1 * float(s) : std::fmaf(d1, float(s), ab);
      }
      a[l] = std::fmaf(d0, ab, a[l]);
    }
  }
  return ((a[0] + a[4]) + (a[2] + a[6])) + ((a[1] + a[5]) + (a[3] + a[7]));
}

// Q2_0 row: 34-byte blocks, codes 0/1/2 = -1/0/+1 (q2.cuh).
float h_row_q2(const uint8_t* row, int64_t nb, const int8_t* q, const uint16_t* d) {
  float a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int64_t b = 0; b < nb; ++b) {
    const uint8_t* blk = row + b * 34;
    const float d0 = h_half(uint16_t(blk[0] | (blk[1] << 8)));
    for (int l = 0; l < 8; ++l) {
      float ab = 0.0f;
      for (int k = 0; k < 4; ++k) {
        int s = 0;
        for (int i = 0; i < 4; ++i) {
          const int j = 32 * k + 4 * l + i;
          const int qq = q[b * kBlock + j];
          const int code = (blk[2 + j / 4] >> (2 * (j % 4))) & 3;
          if (code == 2) s += qq;
          else if (code == 0) s += (qq == -128 ? -128 : -qq);
        }
        const float d1 = h_half(d[b * 4 + k]);
        ab = (k == 0) ? d1 * float(s) : std::fmaf(d1, float(s), ab);
      }
      a[l] = std::fmaf(d0, ab, a[l]);
    }
  }
  return ((a[0] + a[4]) + (a[2] + a[6])) + ((a[1] + a[5]) + (a[3] + a[7]));
}

void h_quant(const float* x, int64_t n, int8_t* q, uint16_t* d) {
  for (int64_t b = 0; b < n / kSub; ++b) {
    float amax = 0.0f;
    for (int j = 0; j < kSub; ++j) amax = std::fmax(amax, std::fabs(x[b * kSub + j]));
    const float dd = amax / 127.0f;
    const float id = dd != 0.0f ? 1.0f / dd : 0.0f;
    d[b] = __half_as_ushort(__float2half_rn(dd));
    for (int j = 0; j < kSub; ++j) q[b * kSub + j] = int8_t(int(std::roundf(x[b * kSub + j] * id)));
  }
}

// ------------------------------------------------------------- inputs -----
struct Rng {
  uint64_t s;
  uint64_t next() {  // splitmix64
    uint64_t z = (s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  double uniform() { return double(next() >> 11) * (1.0 / 9007199254740992.0); }
  double normal() {
    double u1 = uniform(), u2 = uniform();
    if (u1 < 1e-300) u1 = 1e-300;
    return std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586 * u2);
  }
};

uint16_t scale_bits(Rng& r, bool layer) {
  const double v = layer ? std::exp(r.normal() + std::log(0.02)) : std::fabs(r.normal()) * 0.02;
  return __half_as_ushort(__float2half_rn(float(v)));
}

struct Case {
  const char* kernel;  // "q1_0_gemv", "q1_0_gemm_small", "q1_0_gemm_small_noalloc" or "q2_0_gemv"
  int64_t rows, n, nvec;
  bool layer;          // layer-shaped regime: raw quants (with -128), log-normal scales
};

struct Report {
  char* buf;
  size_t cap, len;
  void add(const char* fmt, ...) {
    if (!buf || cap == 0) return;
    va_list ap;
    va_start(ap, fmt);
    int k = vsnprintf(buf + len, cap > len ? cap - len : 0, fmt, ap);
    va_end(ap);
    if (k > 0) len = std::min(cap - 1, len + size_t(k));
  }
};

struct Dev {
  std::vector<void*> ptrs;
  ~Dev() {
    for (void* p : ptrs) cudaFree(p);
  }
  void* get(size_t bytes) {
    void* p = nullptr;
    if (cudaMalloc(&p, bytes < 16 ? 16 : bytes) != cudaSuccess) return nullptr;
    ptrs.push_back(p);
    return p;
  }
};

uint32_t fbits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

// Returns Q1_OK, Q1_MISMATCH or an error.  With `corrupt`, the packed scales
// of one row whose reference output is nonzero are doubled after packing (a
// negative control: the check must then report that row).
int run_case(const Case& c, uint64_t seed, bool corrupt, Report& rep) {
  Rng rng{seed};
  const bool ternary = std::strcmp(c.kernel, "q2_0_gemv") == 0;
  const int64_t nb = c.n / kBlock;
  const int64_t bbytes = ternary ? 34 : kBlockBytes;
  std::vector<uint8_t> blocks(size_t(c.rows * nb * bbytes));
  for (int64_t i = 0; i < c.rows * nb; ++i) {
    uint8_t* blk = &blocks[size_t(i * bbytes)];
    const uint16_t s = scale_bits(rng, c.layer);
    blk[0] = uint8_t(s & 0xff);
    blk[1] = uint8_t(s >> 8);
    for (int j = 2; j < bbytes; ++j) {
      uint8_t v = uint8_t(rng.next());
      if (ternary) v &= uint8_t(~((v & (v >> 1) & 0x55) << 1));  // code 3 -> 1 (a zero weight)
      blk[j] = v;
    }
  }
  std::vector<int8_t> q(size_t(c.nvec * c.n));
  std::vector<uint16_t> d(size_t(c.nvec * c.n / kSub));
  std::vector<float> x;
  if (c.layer) {
    for (auto& v : q) v = int8_t(int(rng.next() % 256) - 128);
    for (size_t i = 0; i < q.size(); i += 37) q[i] = -128;
    for (auto& v : d) v = scale_bits(rng, true);
  } else {
    x.resize(q.size());
    for (auto& v : x) v = float(rng.normal());
    for (int64_t v = 0; v < c.nvec; ++v) h_quant(&x[size_t(v * c.n)], c.n, &q[size_t(v * c.n)], &d[size_t(v * c.n / kSub)]);
  }

  Dev dev;
  const int64_t pbytes = ternary ? q2_0_packed_bytes(c.rows, c.n) : q1_0_packed_bytes(c.rows, c.n);
  uint8_t* d_blocks = static_cast<uint8_t*>(dev.get(blocks.size()));
  void* d_packed = dev.get(size_t(pbytes));
  int8_t* d_q = static_cast<int8_t*>(dev.get(q.size()));
  uint16_t* d_d = static_cast<uint16_t*>(dev.get(d.size() * 2));
  float* d_out = static_cast<float*>(dev.get(size_t(c.nvec * c.rows * 4)));
  float* d_x = x.empty() ? nullptr : static_cast<float*>(dev.get(x.size() * 4));
  if (!d_blocks || !d_packed || !d_q || !d_d || !d_out || (!x.empty() && !d_x))
    return fail(Q1_ERR_NOMEM, "q1_0_verify: device allocation failed");

  if (int e = cuda_status(cudaMemcpy(d_blocks, blocks.data(), blocks.size(), cudaMemcpyHostToDevice), "q1_0_verify copy")) return e;
  if (int e = ternary ? q2_0_pack(d_blocks, c.rows, c.n, d_packed, nullptr)
                      : q1_0_pack(d_blocks, c.rows, c.n, d_packed, nullptr))
    return e;
  if (corrupt && c.nvec == 1) {
    int64_t r0 = c.rows / 2;
    auto ref = [&](int64_t r) {
      const uint8_t* row = &blocks[size_t(r * nb * bbytes)];
      return ternary ? h_row_q2(row, nb, q.data(), d.data()) : h_row(row, nb, q.data(), d.data());
    };
    while (r0 + 1 < c.rows && ref(r0) == 0.0f) ++r0;
    const Layout L = ternary ? layout_q2(c.rows, c.n) : layout_of(c.rows, c.n);
    uint16_t* sc = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(d_packed) + L.bits_bytes);
    for (int64_t b = 0; b < nb; ++b) {
      uint16_t* at = sc + scale_index(r0 / kPanel, b, int(r0 % kPanel), L.nbp);
      uint16_t h = 0;
      if (int e = cuda_status(cudaMemcpy(&h, at, 2, cudaMemcpyDeviceToHost), "q1_0_verify corrupt")) return e;
      if ((h & 0x7c00) != 0 && (h & 0x7c00) < 0x7800) h = uint16_t(h + 0x0400);  // x2, stays finite
      if (int e = cuda_status(cudaMemcpy(at, &h, 2, cudaMemcpyHostToDevice), "q1_0_verify corrupt")) return e;
    }
    rep.add("%s %lldx%lld: scales of row %lld doubled after packing\n", c.kernel, (long long)c.rows,
            (long long)c.n, (long long)r0);
  }
  if (x.empty()) {
    if (int e = cuda_status(cudaMemcpy(d_q, q.data(), q.size(), cudaMemcpyHostToDevice), "q1_0_verify copy")) return e;
    if (int e = cuda_status(cudaMemcpy(d_d, d.data(), d.size() * 2, cudaMemcpyHostToDevice), "q1_0_verify copy")) return e;
  } else {
    if (int e = cuda_status(cudaMemcpy(d_x, x.data(), x.size() * 4, cudaMemcpyHostToDevice), "q1_0_verify copy")) return e;
    if (int e = q8_quantize_act(d_x, c.nvec, c.n, d_q, d_d, nullptr)) return e;
    std::vector<int8_t> gq(q.size());
    std::vector<uint16_t> gd(d.size());
    if (int e = cuda_status(cudaMemcpy(gq.data(), d_q, q.size(), cudaMemcpyDeviceToHost), "q1_0_verify copy")) return e;
    if (int e = cuda_status(cudaMemcpy(gd.data(), d_d, d.size() * 2, cudaMemcpyDeviceToHost), "q1_0_verify copy")) return e;
    for (size_t i = 0; i < q.size(); ++i)
      if (gq[i] != q[i]) {
        rep.add("q8_quantize_act n=%lld: element %zu differs (gpu %d, cpu %d)\n", (long long)c.n, i, gq[i], q[i]);
        return Q1_MISMATCH;
      }
    for (size_t i = 0; i < d.size(); ++i)
      if (gd[i] != d[i]) {
        rep.add("q8_quantize_act n=%lld: scale %zu differs (gpu 0x%04x, cpu 0x%04x)\n", (long long)c.n, i, gd[i], d[i]);
        return Q1_MISMATCH;
      }
  }
  int e = ternary ? q2_0_gemv(d_packed, c.rows, c.n, d_q, d_d, d_out, nullptr)
          : (std::strcmp(c.kernel, "q1_0_gemv") == 0)
              ? q1_0_gemv(d_packed, c.rows, c.n, d_q, d_d, d_out, nullptr)
          : (std::strcmp(c.kernel, "q1_0_gemm_small_noalloc") == 0)  // always the tensor-core kernel
              ? q1_0_gemm_small_noalloc(d_packed, c.rows, c.n, c.nvec, d_q, d_d, d_out, nullptr)
              : q1_0_gemm_small(d_packed, c.rows, c.n, c.nvec, d_q, d_d, d_out, nullptr);
  if (e) return e;
  std::vector<float> out(size_t(c.nvec * c.rows));
  if (int e2 = cuda_status(cudaMemcpy(out.data(), d_out, out.size() * 4, cudaMemcpyDeviceToHost), "q1_0_verify result")) return e2;
  for (int64_t v = 0; v < c.nvec; ++v)
    for (int64_t r = 0; r < c.rows; ++r) {
      const uint8_t* row = &blocks[size_t(r * nb * bbytes)];
      const int8_t* qv = &q[size_t(v * c.n)];
      const uint16_t* dv = &d[size_t(v * c.n / kSub)];
      const float want = ternary ? h_row_q2(row, nb, qv, dv) : h_row(row, nb, qv, dv);
      const float got = out[size_t(v * c.rows + r)];
      if (fbits(want) != fbits(got)) {
        rep.add("%s %lldx%lld nvec=%lld %s: row %lld differs (vector %lld: gpu 0x%08x, cpu 0x%08x)\n", c.kernel,
                (long long)c.rows, (long long)c.n, (long long)c.nvec, c.layer ? "layer-shaped" : "quantized",
                (long long)r, (long long)v, fbits(got), fbits(want));
        return Q1_MISMATCH;
      }
    }
  rep.add("%s %lldx%lld nvec=%lld %s: bit-exact\n", c.kernel, (long long)c.rows, (long long)c.n,
          (long long)c.nvec, c.layer ? "layer-shaped" : "quantized");
  return Q1_OK;
}

// The bounded wait every product kernel uses, on an mbarrier nothing will
// complete: it must give up after about limit_ns and let the kernel return.
__global__ void k_wait_probe(unsigned long long limit_ns, unsigned long long* result) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  const uint64_t t0 = globaltimer();
  const bool got = mbar_wait(smem_addr(&bar), 0u, limit_ns);  // phase 0 never completes
  const uint64_t t1 = globaltimer();
  if (threadIdx.x == 0) {
    result[0] = got ? 1ull : 0ull;
    result[1] = t1 - t0;
  }
}

int run_wait_probe(Report& rep) {
  Dev dev;
  auto* d_res = static_cast<unsigned long long*>(dev.get(16));
  if (!d_res) return fail(Q1_ERR_NOMEM, "q1_0_verify: device allocation failed");
  const unsigned long long limit = 20000000ull;  // 20 ms
  if (int e = launch_plain(k_wait_probe, dim3(1), dim3(32), nullptr, "q1_0_verify wait probe", limit, d_res)) return e;
  unsigned long long res[2] = {0, 0};
  if (int e = cuda_status(cudaMemcpy(res, d_res, 16, cudaMemcpyDeviceToHost), "q1_0_verify wait probe")) return e;
  if (res[0] != 0 || res[1] < limit) {
    rep.add("bounded wait: did not give up as it should (returned %llu after %.2f ms)\n", res[0], res[1] * 1e-6);
    return Q1_MISMATCH;
  }
  rep.add("bounded wait on a barrier nothing completes: gave up after %.2f ms (limit %.0f ms)\n", res[1] * 1e-6,
          limit * 1e-6);
  return Q1_OK;
}

// The product kernels round x * id with adds on the FMA pipe (round_code in
// table.cuh) instead of roundf and a conversion.  Every float t with
// |t| < 2^22 (the kernels' values stay below 127.5) is compared with the
// device's roundf converted to int, low byte.
__global__ void k_round_check(unsigned long long* res, unsigned* first) {
  unsigned long long tested = 0, bad = 0;
  const unsigned long long step = static_cast<unsigned long long>(gridDim.x) * blockDim.x;
  for (unsigned long long i = blockIdx.x * static_cast<unsigned long long>(blockDim.x) + threadIdx.x;
       i < (1ull << 32); i += step) {
    const float t = __uint_as_float(static_cast<uint32_t>(i));
    if (!(fabsf(t) < 4194304.0f)) continue;
    ++tested;
    const uint32_t want = static_cast<uint32_t>(static_cast<int>(roundf(t))) & 0xffu;
    if (round_code(t) != want) {
      ++bad;
      atomicMin(first, static_cast<uint32_t>(i));
    }
  }
  atomicAdd(&res[0], tested);
  atomicAdd(&res[1], bad);
}

int run_round_check(Report& rep) {
  Dev dev;
  auto* d_res = static_cast<unsigned long long*>(dev.get(16));
  auto* d_first = static_cast<unsigned*>(dev.get(4));
  if (!d_res || !d_first) return fail(Q1_ERR_NOMEM, "q1_0_verify: device allocation failed");
  if (int e = cuda_status(cudaMemset(d_res, 0, 16), "q1_0_verify rounding check")) return e;
  if (int e = cuda_status(cudaMemset(d_first, 0xff, 4), "q1_0_verify rounding check")) return e;
  if (int e = launch_plain(k_round_check, dim3(unsigned(num_sms() * 8)), dim3(256), nullptr,
                           "q1_0_verify rounding check", d_res, d_first))
    return e;
  unsigned long long res[2] = {0, 0};
  unsigned first = 0;
  if (int e = cuda_status(cudaMemcpy(res, d_res, 16, cudaMemcpyDeviceToHost), "q1_0_verify rounding check")) return e;
  if (int e = cuda_status(cudaMemcpy(&first, d_first, 4, cudaMemcpyDeviceToHost), "q1_0_verify rounding check"))
    return e;
  if (res[1] != 0) {
    rep.add("q8 rounding by adds: %llu of %llu values differ from roundf, first bits 0x%08x\n", res[1], res[0], first);
    return Q1_MISMATCH;
  }
  rep.add("q8 rounding by adds: all %llu floats with |t| < 2^22 equal roundf\n", res[0]);
  return Q1_OK;
}

}  // namespace
}  // namespace q1

extern "C" int q1_0_verify(int flags, char* report, size_t report_len) {
  using namespace q1;
  Report rep{report, report_len, 0};
  if (report && report_len) report[0] = 0;
  static const Case quick[] = {
      {"q1_0_gemv", 64, 128, 1, true},
      {"q1_0_gemv", 100, 384, 1, false},
      {"q2_0_gemv", 64, 256, 1, true},
  };
  static const Case full[] = {
      {"q1_0_gemv", 64, 128, 1, true},       {"q1_0_gemv", 100, 384, 1, false},   {"q1_0_gemv", 256, 1024, 1, false},
      {"q1_0_gemv", 1000, 4096, 1, true},    {"q1_0_gemv", 33, 14336, 1, true},   {"q1_0_gemv", 4096, 4096, 1, false},
      {"q1_0_gemv", 9999, 1152, 1, true},    {"q1_0_gemm_small", 300, 1024, 3, true},
      {"q1_0_gemm_small", 200, 4096, 16, false}, {"q1_0_gemm_small", 64, 512, 64, true},
      // the tensor-core kernel on a ragged row tile and vector group, and on the layer-shaped
      // regime, whose -128 quants send blocks to its dp4a tables
      {"q1_0_gemm_small_noalloc", 300, 1024, 19, false}, {"q1_0_gemm_small_noalloc", 200, 4096, 16, true},
      {"q2_0_gemv", 64, 128, 1, true},    {"q2_0_gemv", 1000, 4096, 1, false}, {"q2_0_gemv", 33, 14336, 1, true},
      // more panels than one wave of the panel kernel holds: the streaming kernel
      {"q1_0_gemv", 40000, 256, 1, true},    {"q2_0_gemv", 40000, 256, 1, false},
  };
  if (flags & 4) {  // the failure path first; the shape cases after it show the context still works
    if (int e = run_wait_probe(rep)) {
      if (e < 0) return e;
      fail(Q1_MISMATCH, "q1_0_verify: the bounded-wait probe did not give up");
      return e;
    }
  }
  const Case* cs = (flags & 1) ? quick : full;
  const size_t nc = (flags & 1) ? sizeof quick / sizeof quick[0] : sizeof full / sizeof full[0];
  int status = Q1_OK;
  if (!(flags & 1)) {
    const int e = run_round_check(rep);
    if (e < 0) return e;
    if (e == Q1_MISMATCH) status = Q1_MISMATCH;
  }
  for (size_t i = 0; i < nc; ++i) {
    int e = run_case(cs[i], 0x51ED5EEDull + 7919ull * i, (flags & 2) != 0, rep);
    if (e < 0) {
      rep.add("%s\n", q1_last_error());
      return e;
    }
    if (e == Q1_MISMATCH) status = Q1_MISMATCH;
  }
  if (status == Q1_MISMATCH) fail(Q1_MISMATCH, "q1_0_verify: some outputs differ from the host reference");
  return status;
}
