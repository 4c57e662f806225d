// Accumulation error of the encoder's tensor-core sums (tcgen05.mma kind::tf32, M = 128, N = 64,
// K = 8, operands K-major in shared memory without swizzle, accumulators in tensor memory).
// One CTA of 128 threads per trial.  A full fp32 per-vector operand a is split into tf32 parts
// hi = rna(a), lo = rna(a - hi), and the parts' MMAs accumulate into one column, as the encoder
// does:
//   plain sums     a . b over 8 terms (2 MMAs), a signed or positive, b one of the codebook
//                  operand kinds: g^2 of {8, 25, 43}, {8, 25, 43}, ternary, |ternary|
//   deferred sums  w . h + sig (w/4) . g over 8 + 8 terms (4 MMAs), w >= 0, g ternary, h = |g|
//   split sums     a . h with h = g^2 of integers g up to 127 (up to 14 significant bits) split
//                  into exact tf32 parts hi + lo: a hi . h hi + a lo . h hi + a hi . h lo +
//                  a lo . h lo (4 MMAs)
//   encoder operands  plain sums whose a is the encoder's own per-vector operand (w, or
//                  -2 w t) for blocks drawn like the bench weight and importance
// Each result is compared with the exact value in fp64; the program prints the worst
// |D - exact| / sum |terms| in units u = 2^-24 per operand kind.  All waits are bounded.
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <cmath>
#include <vector>
#include <random>
#include <cuda_runtime.h>

#define M 128
#define N 64
#define K 8

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t gtimer() { uint64_t t; asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)); return t; }
__device__ __forceinline__ bool mbar_wait(uint64_t *m, uint32_t par) {
  const uint64_t t0 = gtimer();
  while (true) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(smem_u32(m)), "r"(par) : "memory");
    if (ok) return true;
    if (gtimer() - t0 > 1000000000ull) return false;
  }
}
__device__ __forceinline__ float tf32(float x) { uint32_t r; asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x)); return __uint_as_float(r); }

// canonical K-major, no swizzle: core matrix = 8 rows x 16 bytes (4 elements), 128 contiguous bytes;
// along K: core matrices LBO = 128 bytes apart; along M/N: groups of 8 rows SBO = 256 bytes apart.
__host__ __device__ __forceinline__ int kmaj_off(int row, int k) {  // in floats
  return (row >> 3) * 64 + (k >> 2) * 32 + (row & 7) * 4 + (k & 3);
}
__device__ __forceinline__ uint64_t sdesc(const void *base, uint32_t lbo, uint32_t sbo) {
  const uint64_t a = smem_u32(base);
  return ((a >> 4) & 0x3fff) | ((uint64_t)((lbo >> 4) & 0x3fff) << 16) | ((uint64_t)((sbo >> 4) & 0x3fff) << 32) |
         (1ull << 46);
}

__global__ void __launch_bounds__(128, 1) probe(const float *A, const float *B, const float *B2, float *D, int nsplit,
                                                int *err, uint32_t lbo, uint32_t sbo, float sig, int hsplit) {
  __shared__ __align__(1024) float sA[4][M * K];   // w hi, w lo, sig w/4 hi, sig w/4 lo
  __shared__ __align__(1024) float sB[2][N * K];    // h, g
  __shared__ uint64_t mbar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // operands -> shared memory (canonical layout), A split into tf32 parts
  for (int i = tid; i < M * K; i += blockDim.x) {
    const int r = i / K, k = i % K;
    const float a = A[i];
    const float h = tf32(a), l = tf32(a - h);
    sA[0][kmaj_off(r, k)] = h;
    sA[1][kmaj_off(r, k)] = l;
    sA[2][kmaj_off(r, k)] = sig * 0.25f * h;
    sA[3][kmaj_off(r, k)] = sig * 0.25f * l;
  }
  for (int i = tid; i < N * K; i += blockDim.x) {
    sB[0][kmaj_off(i / K, i % K)] = B[i];
    sB[1][kmaj_off(i / K, i % K)] = B2[i];
  }
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&mbar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)), "r"(64));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
  if (tid == 0) {
    for (int s = 0; s < nsplit; s++) {
      const uint64_t bdesc = sdesc(sB[s < 2 ? 0 : 1], lbo, sbo);
      const uint64_t adesc = sdesc(sA[hsplit ? (s & 1) : s], lbo, sbo);
      const uint32_t acc = s > 0;
      asm volatile("{ .reg .pred p; setp.ne.u32 p, %4, 0; tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p; }"
                   ::"r"(tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&mbar))
                 : "memory");
  }
  const bool ok = mbar_wait(&mbar, 0);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (!ok) { if (tid == 0) atomicOr(err, 1); }
  else {
    // each warp reads its 32 lanes (rows 32w..32w+31), 16 columns at a time
    for (int c0 = 0; c0 < N; c0 += 16) {
      uint32_t r[16];
      const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0;
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                   : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                     "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                   : "r"(taddr));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      for (int j = 0; j < 16; j++) D[(32 * warp + lane) * N + c0 + j] = __uint_as_float(r[j]);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(64));
}

static double worst_of(const std::vector<float> &D, const std::vector<double> &ex, const std::vector<double> &ab) {
  double mx = 0;
  for (size_t i = 0; i < D.size(); i++)
    if (ab[i] > 0) mx = std::max(mx, std::fabs((double)D[i] - ex[i]) / ab[i]);
  return mx / 5.9604644775390625e-08;
}

int main() {
  std::mt19937 rng(7);
  std::normal_distribution<float> nd(0.f, 1.f);
  std::uniform_int_distribution<int> ud(0, 2);
  const float vals[3] = {8.f, 25.f, 43.f};
  std::vector<float> A(M * K), H(N * K), Gv(N * K), D(M * N);
  std::vector<double> ex(M * N), ab(M * N);
  float *dA, *dH, *dG, *dD; int *derr;
  cudaMalloc(&dA, A.size() * 4); cudaMalloc(&dH, H.size() * 4); cudaMalloc(&dG, Gv.size() * 4);
  cudaMalloc(&dD, D.size() * 4); cudaMalloc(&derr, 4);
  auto launch = [&](int nsplit, float sig, int hsplit = 0) -> bool {
    cudaMemcpy(dA, A.data(), A.size() * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(dH, H.data(), H.size() * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(dG, Gv.data(), Gv.size() * 4, cudaMemcpyHostToDevice);
    cudaMemset(derr, 0, 4); cudaMemset(dD, 0, D.size() * 4);
    probe<<<1, 128>>>(dA, dH, dG, dD, nsplit, derr, 128, 256, sig, hsplit);
    cudaError_t e = cudaDeviceSynchronize();
    int herr = 0; cudaMemcpy(&herr, derr, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess || herr) { printf("error %s timeout=%d\n", cudaGetErrorString(e), herr); return false; }
    cudaMemcpy(D.data(), dD, D.size() * 4, cudaMemcpyDeviceToHost);
    return true;
  };
  // plain sums: a . b, 8 terms, a in four distributions, b in the four codebook operand kinds
  double plain[4] = {};
  for (int trial = 0; trial < 160; trial++) {
    const int bk = trial % 4, ak = (trial / 4) % 4;
    for (int m = 0; m < M; m++)
      for (int k = 0; k < K; k++) {
        float a;
        if (ak == 0) a = nd(rng) * std::exp(nd(rng));
        else if (ak == 1) a = std::exp(3.0f * nd(rng));
        else if (ak == 2) { const float b = std::exp(nd(rng)); a = (k & 1) ? -A[m * K + k - 1] * (1.0f + 1e-3f * nd(rng)) : b; }
        else a = 1.0f + std::fabs(nd(rng)) * 0.3f;
        A[m * K + k] = a;
      }
    for (auto &b : H) {
      const int d = ud(rng);
      b = bk == 0 ? vals[d] * vals[d] : bk == 1 ? vals[d] : bk == 2 ? (float)(d - 1) : (float)std::abs(d - 1);
    }
    if (!launch(2, 1.0f)) return 1;
    for (int m = 0; m < M; m++)
      for (int n = 0; n < N; n++) {
        double e = 0, s = 0;
        for (int k = 0; k < K; k++) { const double t = (double)A[m * K + k] * H[n * K + k]; e += t; s += std::fabs(t); }
        ex[m * N + n] = e; ab[m * N + n] = s;
      }
    plain[bk] = std::max(plain[bk], worst_of(D, ex, ab));
  }
  const char *bn[4] = {"g2", "g", "ternary", "absternary"};
  for (int bk = 0; bk < 4; bk++) printf("plain %s %.3f\n", bn[bk], plain[bk]);
  // deferred sums: w . h + sig (w/4) . g, w >= 0 in four distributions
  double dfr[2] = {};
  for (int trial = 0; trial < 160; trial++) {
    const int ak = trial % 4;
    for (auto &a : A)
      a = ak == 0 ? std::fabs(nd(rng)) * std::exp(nd(rng)) : ak == 1 ? std::exp(3.0f * nd(rng))
        : ak == 2 ? 1.0f + std::fabs(nd(rng)) * 0.3f : std::exp(nd(rng));
    for (int i = 0; i < N * K; i++) { const int d = ud(rng) - 1; Gv[i] = (float)d; H[i] = (float)std::abs(d); }
    for (int si = 0; si < 2; si++) {
      const float sig = si ? -1.0f : 1.0f;
      if (!launch(4, sig)) return 1;
      for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++) {
          double e = 0, s = 0;
          for (int k = 0; k < K; k++) {
            const double w = A[m * K + k], h = H[n * K + k], g = Gv[n * K + k];
            e += w * h + sig * 0.25 * w * g;
            s += std::fabs(w * h) + std::fabs(0.25 * w * g);
          }
          ex[m * N + n] = e; ab[m * N + n] = s;
        }
      dfr[si] = std::max(dfr[si], worst_of(D, ex, ab));
    }
  }
  printf("deferred plus %.3f\n", dfr[0]);
  printf("deferred minus %.3f\n", dfr[1]);
  // split sums: h = g^2 for integers g in [1, 127] (a third of them 47, 101 or 127), as hi + lo
  std::uniform_int_distribution<int> gd(1, 127), pick(0, 5);
  const int wide[3] = {47, 101, 127};
  auto tf32_host = [](float x) {  // round to nearest (ties away), 10 explicit mantissa bits
    uint32_t b; std::memcpy(&b, &x, 4); b = (b + 0x1000u) & ~0x1fffu; std::memcpy(&x, &b, 4); return x;
  };
  double spl = 0;
  std::vector<double> Hx(N * K);
  for (int trial = 0; trial < 160; trial++) {
    const int ak = trial % 4;
    for (int m = 0; m < M; m++)
      for (int k = 0; k < K; k++) {
        float a;
        if (ak == 0) a = nd(rng) * std::exp(nd(rng));
        else if (ak == 1) a = std::exp(3.0f * nd(rng));
        else if (ak == 2) { const float b = std::exp(nd(rng)); a = (k & 1) ? -A[m * K + k - 1] * (1.0f + 1e-3f * nd(rng)) : b; }
        else a = 1.0f + std::fabs(nd(rng)) * 0.3f;
        A[m * K + k] = a;
      }
    for (int i = 0; i < N * K; i++) {
      const int p = pick(rng);
      const int g = p < 2 ? wide[p] : p == 2 ? 127 : gd(rng);
      const float h = (float)(g * g), hi = tf32_host(h);
      H[i] = hi; Gv[i] = h - hi; Hx[i] = (double)g * g;
    }
    if (!launch(4, 1.0f, 1)) return 1;
    for (int m = 0; m < M; m++)
      for (int n = 0; n < N; n++) {
        double e = 0, s = 0;
        for (int k = 0; k < K; k++) { const double t = (double)A[m * K + k] * Hx[n * K + k]; e += t; s += std::fabs(t); }
        ex[m * N + n] = e; ab[m * N + n] = s;
      }
    spl = std::max(spl, worst_of(D, ex, ab));
  }
  printf("split g2wide %.3f\n", spl);
  // the encoder's own operands: for a block of 256 weights drawn like the bench weight (Student-t,
  // 4 degrees of freedom) with importance drawn like the bench's (root mean square over 4096
  // activation rows of N(0, 1) times a log-normal column scale), the per-vector operands are w and
  // nw2 = -2 w t, with t the magnitude in grid units under a random choice c: |x| / (d (2c+1)/8),
  // d = amax / 166.625 (the IQ2 anchor).  Both go against the four codebook operand kinds.
  std::student_t_distribution<float> td(4.0f);
  std::uniform_int_distribution<int> cd(0, 15);
  double enc = 0;
  for (int trial = 0; trial < 160; trial++) {
    const int bk = trial % 4, wk = (trial / 4) % 2;
    for (int blk = 0; blk < M * K / 256; blk++) {
      float x[256], amax = 0.f;
      for (int i = 0; i < 256; i++) { x[i] = 0.02f * td(rng); amax = std::max(amax, std::fabs(x[i])); }
      const float d = amax / 166.625f;
      for (int i = 0; i < 256; i++) {
        const float sc = std::exp(nd(rng));
        double ss = 0;
        for (int r = 0; r < 4096; r += 64) { const double v = nd(rng) * sc; ss += v * v; }  // 64 of the rows
        const float w = (float)std::sqrt(ss / 64.0);
        const float t = std::fabs(x[i]) / (d * (2 * cd(rng) + 1) / 8.0f);
        A[blk * 256 + i] = wk ? -2.0f * w * t : w;
      }
    }
    for (auto &b : H) {
      const int dd = ud(rng);
      b = bk == 0 ? vals[dd] * vals[dd] : bk == 1 ? vals[dd] : bk == 2 ? (float)(dd - 1) : (float)std::abs(dd - 1);
    }
    if (!launch(2, 1.0f)) return 1;
    for (int m = 0; m < M; m++)
      for (int n = 0; n < N; n++) {
        double e = 0, s = 0;
        for (int k = 0; k < K; k++) { const double t = (double)A[m * K + k] * H[n * K + k]; e += t; s += std::fabs(t); }
        ex[m * N + n] = e; ab[m * N + n] = s;
      }
    enc = std::max(enc, worst_of(D, ex, ab));
  }
  printf("plain encoder-operands %.3f\n", enc);
  return 0;
}
