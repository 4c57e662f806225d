// Device-side definitions shared by the library's kernels: format traits, payload bit fields,
// the super-block anchor and the sign rule.  Layouts and rules are the ones documented in
// include/iq.h (PR #2513 IQ2_XXS / IQ2_S / IQ1_M commit texts; PR #3157 choices).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/iq.h"

namespace iqk {

constexpr float kU = 5.9604644775390625e-08f;  // 2^-24, unit roundoff of fp32
// Rounding bound of the fp32 expanded-form scores, in units of weighted squared error: a decision
// between two candidates (or two choices) of errors E1 <= E2 over a unit with sum w t^2 = Cs is
// trusted only when the computed gap exceeds kMargin * (2 Cs + E1 + E2).  The fp32 error of one
// score is below 44u Cs + 35u E for IQ2 and about 60u Cs + 50u E for IQ1 (FMA chains of length 8,
// shifted IQ1 sums), so 128u leaves a factor of two.
constexpr float kMargin = 128.0f * kU;

template <int F> struct Fmt;
template <> struct Fmt<IQ2_XXS> { static constexpr int BB = 66, G = 8, C = 16, N = 256, VPG = 4, IQ1 = 0, PAR = 1; };
template <> struct Fmt<IQ2_XS>  { static constexpr int BB = 74, G = 16, C = 16, N = 512, VPG = 2, IQ1 = 0, PAR = 1; };
template <> struct Fmt<IQ2_S>   { static constexpr int BB = 82, G = 16, C = 16, N = 1024, VPG = 2, IQ1 = 0, PAR = 0; };
template <> struct Fmt<IQ1_S>   { static constexpr int BB = 50, G = 8, C = 16, N = 2048, VPG = 4, IQ1 = 1, PAR = 0; };
template <> struct Fmt<IQ1_M>   { static constexpr int BB = 56, G = 16, C = 8, N = 2048, VPG = 2, IQ1 = 1, PAR = 0; };

__host__ __device__ inline int fmt_block_bytes(int f) {
  return f == IQ2_XXS ? 66 : f == IQ2_XS ? 74 : f == IQ2_S ? 82 : f == IQ1_S ? 50 : 56;
}

// ---------------------------------------------------------------------------------------------
// Payload bit fields.  A block is at most 82 bytes; a warp assembles it in 24 shared 32-bit words.
struct Bits { int pos, width; };

// Field positions for vector g (0..31) and choice group cg.
template <int F> __device__ __forceinline__ Bits f_d16() { return {0, 16}; }
template <int F> __device__ __forceinline__ Bits f_idx_lo(int g) {
  if (F == IQ2_XXS) return {(2 + 8 * (g >> 2) + (g & 3)) * 8, 8};
  if (F == IQ2_XS) return {(2 + 2 * g) * 8, 9};
  if (F == IQ2_S || F == IQ1_S) return {(2 + g) * 8, 8};
  return {g * 8, 8};  // IQ1_M
}
template <int F> __device__ __forceinline__ Bits f_idx_hi(int g) {
  if (F == IQ2_S) return {(66 + (g >> 2)) * 8 + 2 * (g & 3), 2};
  if (F == IQ1_S) return {(34 + 2 * (g >> 2)) * 8 + 3 * (g & 3), 3};
  if (F == IQ1_M) return {(32 + (g >> 1)) * 8 + 4 * (g & 1), 3};
  return {0, 0};
}
template <int F> __device__ __forceinline__ Bits f_sign(int g) {
  if (F == IQ2_XXS) return {(6 + 8 * (g >> 2)) * 8 + 7 * (g & 3), 7};
  if (F == IQ2_XS) return {(2 + 2 * g) * 8 + 9, 7};
  if (F == IQ2_S) return {(34 + g) * 8, 8};
  return {0, 0};
}
template <int F> __device__ __forceinline__ Bits f_dbit_vec(int g) {  // IQ1_M only
  return {(32 + (g >> 1)) * 8 + 4 * (g & 1) + 3, 1};
}
template <int F> __device__ __forceinline__ Bits f_scale(int cg) {
  if (F == IQ2_XXS) return {(6 + 8 * cg) * 8 + 28, 4};
  if (F == IQ2_XS) return {(66 + (cg >> 1)) * 8 + 4 * (cg & 1), 4};
  if (F == IQ2_S) return {(74 + (cg >> 1)) * 8 + 4 * (cg & 1), 4};
  if (F == IQ1_S) return {(34 + 2 * cg) * 8 + 12, 3};
  return {(48 + 2 * (cg >> 2)) * 8 + 3 * (cg & 3), 3};  // IQ1_M
}
template <int F> __device__ __forceinline__ Bits f_dbit_grp(int cg) {  // IQ1_S only
  return {(34 + 2 * cg) * 8 + 15, 1};
}
template <int F> __device__ __forceinline__ Bits f_d16_nib(int k) {  // IQ1_M only
  return {(48 + 2 * k) * 8 + 12, 4};
}

// OR `value` (width <= 16 bits) into a shared bit buffer of 32-bit words.
__device__ __forceinline__ void put_bits(uint32_t *buf, Bits b, uint32_t value) {
  if (b.width == 0) return;
  value &= (1u << b.width) - 1u;
  int w = b.pos >> 5, o = b.pos & 31;
  atomicOr(&buf[w], value << o);
  if (o + b.width > 32) atomicOr(&buf[w + 1], value >> (32 - o));
}
__device__ __forceinline__ uint32_t get_bits(const uint8_t *p, Bits b) {
  if (b.width == 0) return 0;
  int byte = b.pos >> 3, o = b.pos & 7;
  uint32_t v = (uint32_t)p[byte];                       // read only the bytes the field spans
  if (o + b.width > 8) v |= (uint32_t)p[byte + 1] << 8;
  if (o + b.width > 16) v |= (uint32_t)p[byte + 2] << 16;
  return (v >> o) & ((1u << b.width) - 1u);
}
// Byte-wise read-modify-write of one field (single thread; used by the rescoring pass).
__device__ __forceinline__ void set_bits_bytes(uint8_t *p, Bits b, uint32_t value) {
  for (int i = 0; i < b.width; i++) {
    int bit = b.pos + i;
    uint8_t m = (uint8_t)(1u << (bit & 7));
    if ((value >> i) & 1u) p[bit >> 3] |= m; else p[bit >> 3] &= (uint8_t)~m;
  }
}

// ---------------------------------------------------------------------------------------------
// Loads of one 8-value vector.
__device__ __forceinline__ void load8(const float *p, float *v) {
  float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float *v) {
  uint4 r = __ldg(reinterpret_cast<const uint4 *>(p));
  uint32_t u[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int k = 0; k < 4; k++) {
    v[2 * k] = __uint_as_float(u[k] << 16);
    v[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
  }
}

__device__ __forceinline__ bool finite8(const float *v) {
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 8; i++) ok &= isfinite(v[i]);
  return ok;
}

// ---------------------------------------------------------------------------------------------
// Super-block anchor, one warp per block (lane l holds values 8l..8l+7).  Every operation is an
// explicitly rounded IEEE fp32 operation, so the result does not depend on compiler contraction.
template <int F>
__device__ __forceinline__ float anchor_scale(const float *x) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; i++) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  float d;
  if (F == IQ1_M) {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) s = __fadd_rn(s, __fmul_rn(x[i], x[i]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    float rms = __fsqrt_rn(__fdiv_rn(s, 256.0f));
    float p2r = __fdiv_rn(amax, rms);
    float r = __fadd_rn(0.58f, __fmul_rn(0.035f, p2r));
    r = fminf(fmaxf(r, 0.65f), 0.95f);
    d = amax == 0.0f ? 0.0f : __fdiv_rn(__fmul_rn(r, amax), 15.0f);
  } else if (F == IQ1_S) {
    d = __fdiv_rn(__fmul_rn(0.61f, amax), 15.0f);
  } else {
    d = __fdiv_rn(amax, 166.625f);
  }
  return fminf(d, 65504.0f);
}

__device__ __forceinline__ uint16_t half_bits_rn(float d) { return __half_as_ushort(__float2half_rn(d)); }
__device__ __forceinline__ float half_bits_to_float(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// Sign rule: returns the 8-bit sign mask and writes t (the value the magnitude grid must match:
// |x_i| for kept signs, -|x_i| for the element whose sign bit was flipped to restore even parity).
template <int F>
__device__ __forceinline__ int sign_rule(const float *x, const float *w, float *t) {
  int m = 0;
#pragma unroll
  for (int i = 0; i < 8; i++) m |= (x[i] < 0.0f ? 1 : 0) << i;
  if (Fmt<F>::PAR && (__popc(m) & 1)) {
    int best = 0;
    float bk = __fmul_rn(w[0], __fmul_rn(x[0], x[0]));
#pragma unroll
    for (int i = 1; i < 8; i++) {
      float k = __fmul_rn(w[i], __fmul_rn(x[i], x[i]));
      if (k < bk) { bk = k; best = i; }
    }
    m ^= 1 << best;
  }
#pragma unroll
  for (int i = 0; i < 8; i++) t[i] = ((m >> i) & 1) ? -x[i] : x[i];
  return m;
}

__device__ __forceinline__ int parity7(int s) { return __popc(s & 0x7f) & 1; }

// ---------------------------------------------------------------------------------------------
// mbarrier and bulk-copy (TMA engine) helpers.  Every wait is bounded by the global timer, so a
// copy that never lands makes the caller report IQ_STATUS_TIMEOUT instead of hanging.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *m, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(m)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t *m, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(m)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *m) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(m)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *m, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(m)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait with a suspend-time hint: a thread whose phase is not complete sleeps (up to the hint,
// waking early when the phase completes) instead of spinning on issue slots other warps need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *m, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(m)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}
// Waits for the phase of parity `parity` to complete; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *m, uint32_t parity) {
  if (mbar_try_wait(m, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_sleep(m, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}
// Untiled bulk copy global -> this CTA's shared memory (16-byte aligned addresses and size).
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(mbar))
      : "memory");
}
// Tiled 2-D tensor copy (box of the tensor map) at element coordinates (x inner, y outer) into
// this CTA's shared memory.  x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x, int y, uint64_t *mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(mbar))
      : "memory");
}

}  // namespace iqk
