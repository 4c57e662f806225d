// Decoder: payload blocks -> values (PR #2513: value rule of each format; layouts in iq.h).
// One warp decodes one 256-value block per step; lane g reads vector g's fields and writes its
// 8 values as two 16-byte stores (fp32) or one (bf16), so a warp writes 1 KiB (fp32) contiguously.
// Every decoded value is an exact product in fp32, so the result is bit-identical to any correct
// evaluation of the value rule.
#include "iq_common.cuh"

namespace iqk {

template <int F>
__device__ __forceinline__ void decode_vector(const uint8_t *p, const float *__restrict__ grid, int g, float *q) {
  constexpr int VPG = Fmt<F>::VPG;
  uint32_t d16;
  if (F == IQ1_M) {
    d16 = 0;
#pragma unroll
    for (int k = 0; k < 4; k++) d16 |= get_bits(p, f_d16_nib<F>(k)) << (4 * k);
  } else {
    d16 = get_bits(p, f_d16<F>());
  }
  const float d = half_bits_to_float((uint16_t)d16);
  const int cg = g / VPG;
  const int s = (int)get_bits(p, f_scale<F>(cg));
  const Bits lo = f_idx_lo<F>(g);
  const int idx = (int)(get_bits(p, lo) | (get_bits(p, f_idx_hi<F>(g)) << lo.width));
  float gv[8];
  load8(grid + 8 * idx, gv);
  if (!Fmt<F>::IQ1) {
    int sg = (int)get_bits(p, f_sign<F>(g));
    if (Fmt<F>::PAR) sg |= parity7(sg) << 7;
    const float dl = __fmul_rn(__fmul_rn(d, (float)(2 * s + 1)), 0.125f);
#pragma unroll
    for (int i = 0; i < 8; i++) {
      float v = __fmul_rn(dl, gv[i]);
      q[i] = ((sg >> i) & 1) ? -v : v;
    }
  } else {
    const int db = F == IQ1_S ? (int)get_bits(p, f_dbit_grp<F>(cg)) : (int)get_bits(p, f_dbit_vec<F>(g));
    const float delta = db ? -0.125f : 0.125f;
    const float dl = __fmul_rn(d, (float)(2 * s + 1));
#pragma unroll
    for (int i = 0; i < 8; i++) q[i] = __fmul_rn(dl, __fadd_rn(gv[i], delta));
  }
}

__device__ __forceinline__ void store8(float *o, const float *q) {
  reinterpret_cast<float4 *>(o)[0] = make_float4(q[0], q[1], q[2], q[3]);
  reinterpret_cast<float4 *>(o)[1] = make_float4(q[4], q[5], q[6], q[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16 *o, const float *q) {
  uint32_t u[4];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    __nv_bfloat162 h = __floats2bfloat162_rn(q[2 * k], q[2 * k + 1]);
    u[k] = *reinterpret_cast<uint32_t *>(&h);
  }
  *reinterpret_cast<uint4 *>(o) = make_uint4(u[0], u[1], u[2], u[3]);
}

template <int F, typename TOut>
__global__ void __launch_bounds__(256) decode_kernel(const uint8_t *__restrict__ payload, int64_t nblocks,
                                                     const float *__restrict__ grid, TOut *__restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t b = warp; b < nblocks; b += nwarps) {
    float q[8];
    decode_vector<F>(payload + b * Fmt<F>::BB, grid, lane, q);
    store8(out + b * 256 + lane * 8, q);
  }
}

template <int F>
static int launch_decode(const uint8_t *payload, int64_t nblocks, const float *grid, void *out, iq_dtype dt,
                         cudaStream_t st) {
  if (nblocks == 0) return IQ_OK;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t want = (nblocks + 7) / 8;
  int grid_x = (int)(want < (int64_t)sms * 16 ? want : (int64_t)sms * 16);
  if (dt == IQ_F32)
    decode_kernel<F, float><<<grid_x, 256, 0, st>>>(payload, nblocks, grid, (float *)out);
  else
    decode_kernel<F, __nv_bfloat16><<<grid_x, 256, 0, st>>>(payload, nblocks, grid, (__nv_bfloat16 *)out);
  return cudaPeekAtLastError() == cudaSuccess ? IQ_OK : IQ_ERR_CUDA;
}

}  // namespace iqk

using namespace iqk;

extern "C" int iq_decode(iq_format f, const uint8_t *payload, int64_t rows, int64_t cols, const float *grid,
                         void *out, iq_dtype out_dtype, void *stream) {
  if ((unsigned)f > IQ1_M || rows < 0 || cols <= 0 || cols % 256) return IQ_ERR_ARG;
  if (out_dtype != IQ_F32 && out_dtype != IQ_BF16) return IQ_ERR_ARG;
  const int64_t nb = rows * (cols / 256);
  if (nb > 0 && (!payload || !grid || !out)) return IQ_ERR_ARG;
  if (((uintptr_t)grid & 15) || ((uintptr_t)out & 15)) return IQ_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  switch (f) {
    case IQ2_XXS: return launch_decode<IQ2_XXS>(payload, nb, grid, out, out_dtype, st);
    case IQ2_XS: return launch_decode<IQ2_XS>(payload, nb, grid, out, out_dtype, st);
    case IQ2_S: return launch_decode<IQ2_S>(payload, nb, grid, out, out_dtype, st);
    case IQ1_S: return launch_decode<IQ1_S>(payload, nb, grid, out, out_dtype, st);
    default: return launch_decode<IQ1_M>(payload, nb, grid, out, out_dtype, st);
  }
}
