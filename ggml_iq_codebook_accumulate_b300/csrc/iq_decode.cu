// Decoder: payload blocks -> values (PR #2513: value rule of each format; layouts in iq.h).
//
// One warp decodes one 256-value block per step.  The block's bytes are staged in the warp's
// registers with one coalesced 32-bit load per lane (the aligned 128-byte window that holds the
// block); every field is then read with two shuffles and a funnel shift, so each lane issues one
// payload load instead of one load per field.  Lane l produces two runs of 4 values: values 4l..4l+3
// and 128+4l..128+4l+3 (half h = l & 1 of vectors l/2 and 16 + l/2), so each store instruction of
// the warp writes one contiguous 512-byte (fp32) or 256-byte (bf16) span.  Every decoded value is an
// exact product in fp32, so the result is bit-identical to any correct evaluation of the rule.
#include "iq_common.cuh"

namespace iqk {

// Field (pos, width) of the block whose first byte is `sh` bits into the staged window.
__device__ __forceinline__ uint32_t wbits(uint32_t wv, int sh, Bits b) {
  if (b.width == 0) return 0;
  const int p = sh + b.pos;
  const uint32_t lo = __shfl_sync(0xffffffffu, wv, p >> 5);
  const uint32_t hi = __shfl_sync(0xffffffffu, wv, (p >> 5) + 1);
  return __funnelshift_r(lo, hi, p & 31) & ((1u << b.width) - 1u);
}

// The 4 values of half `h` of vector g (values 8g + 4h .. 8g + 4h + 3).
template <int F>
__device__ __forceinline__ void decode_half(uint32_t wv, int sh, const float *__restrict__ grid, int g, int h,
                                            float *q) {
  constexpr int VPG = Fmt<F>::VPG;
  uint32_t d16;
  if (F == IQ1_M) {
    d16 = 0;
#pragma unroll
    for (int k = 0; k < 4; k++) d16 |= wbits(wv, sh, f_d16_nib<F>(k)) << (4 * k);
  } else {
    d16 = wbits(wv, sh, f_d16<F>());
  }
  const float d = half_bits_to_float((uint16_t)d16);
  const int cg = g / VPG;
  const int s = (int)wbits(wv, sh, f_scale<F>(cg));
  const Bits lo = f_idx_lo<F>(g);
  const int idx = (int)(wbits(wv, sh, lo) | (wbits(wv, sh, f_idx_hi<F>(g)) << lo.width));
  const float4 gv = __ldg(reinterpret_cast<const float4 *>(grid + 8 * idx + 4 * h));
  const float gg[4] = {gv.x, gv.y, gv.z, gv.w};
  if (!Fmt<F>::IQ1) {
    int sg = (int)wbits(wv, sh, f_sign<F>(g));
    if (Fmt<F>::PAR) sg |= parity7(sg) << 7;
    const float dl = __fmul_rn(__fmul_rn(d, (float)(2 * s + 1)), 0.125f);
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const float v = __fmul_rn(dl, gg[i]);
      q[i] = ((sg >> (4 * h + i)) & 1) ? -v : v;
    }
  } else {
    const int db = F == IQ1_S ? (int)wbits(wv, sh, f_dbit_grp<F>(cg)) : (int)wbits(wv, sh, f_dbit_vec<F>(g));
    const float delta = db ? -0.125f : 0.125f;
    const float dl = __fmul_rn(d, (float)(2 * s + 1));
#pragma unroll
    for (int i = 0; i < 4; i++) q[i] = __fmul_rn(dl, __fadd_rn(gg[i], delta));
  }
}

__device__ __forceinline__ void store4(float *o, const float *q) {
  *reinterpret_cast<float4 *>(o) = make_float4(q[0], q[1], q[2], q[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16 *o, const float *q) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(q[0], q[1]), b = __floats2bfloat162_rn(q[2], q[3]);
  *reinterpret_cast<uint2 *>(o) = make_uint2(*reinterpret_cast<const uint32_t *>(&a),
                                             *reinterpret_cast<const uint32_t *>(&b));
}

template <int F, typename TOut>
__global__ void __launch_bounds__(256) decode_kernel(const uint8_t *__restrict__ payload, int64_t nblocks,
                                                     const float *__restrict__ grid, TOut *__restrict__ out) {
  constexpr int BB = Fmt<F>::BB;
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t total = nblocks * BB;
  // windows are aligned on the absolute address: with the payload at m bytes past a 4-byte
  // boundary, the window of a block starts at the boundary below it (the bytes before the payload
  // that share its first word are read and shifted out; they lie in the same allocation, whose
  // start is aligned), and any word reaching past the end is read byte by byte
  const int m = (int)((uintptr_t)payload & 3);
  const uint8_t *p0 = payload - m;
  const int64_t end = total + m;
  const int g0 = lane >> 1, g1 = 16 + (lane >> 1), h = lane & 1;
  for (int64_t b = warp; b < nblocks; b += nwarps) {
    const int64_t base = b * BB + m, a0 = base & ~(int64_t)3;
    const int64_t at = a0 + 4 * lane;
    uint32_t wv = 0;
    if (at + 4 <= end) {
      wv = __ldg(reinterpret_cast<const uint32_t *>(p0 + at));
    } else {
#pragma unroll
      for (int k = 0; k < 4; k++)
        if (at + k < end && at + k >= m) wv |= (uint32_t)p0[at + k] << (8 * k);
    }
    const int sh = (int)(base - a0) * 8;
    float q0[4], q1[4];
    decode_half<F>(wv, sh, grid, g0, h, q0);
    decode_half<F>(wv, sh, grid, g1, h, q1);
    store4(out + b * 256 + 4 * lane, q0);
    store4(out + b * 256 + 128 + 4 * lane, q1);
  }
}

template <int F>
static int launch_decode(const uint8_t *payload, int64_t nblocks, const float *grid, void *out, iq_dtype dt,
                         cudaStream_t st) {
  if (nblocks == 0) return IQ_OK;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (nblocks + 7) / 8;
  const int grid_x = (int)(want < (int64_t)sms * 16 ? want : (int64_t)sms * 16);
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
