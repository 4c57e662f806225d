// imatrix statistic: routed per-expert sums of squared activations and token counts
// ("Add imatrix calibration for the GGML formats ...", What imatrix does: one statistic per
// routed expert over the tokens routed to it, rows squared 1,024 at a time; "MoE expert coverage
// in imatrix calibration", Facts: x^2 added only to the token's top-k experts, a per-expert token
// count, non-finite sums checked only for touched experts, count 0 -> weight 1).
//
// Two kernels per call:
//  route       one CTA per chunk: a bitmap [E][rows/32] of which chunk rows each expert receives
//              (a token's ids are a set), per-chunk counts, and an expert order by descending count;
//  accumulate  one CTA per 64-column tile walks the chunks in order.  Each chunk is streamed through
//              shared memory in sub-tiles (cp.async, double buffered); warp w owns a fixed set of
//              experts (dealt from the count order so heavy and light experts mix) and, for each,
//              walks the set bits of its bitmap in ascending row order adding x*x to a register
//              accumulator per column (one rounded multiply and one rounded add).  After the chunk
//              the partial sums are added to in_sum2 once, in chunk order.  This is exactly the
//              sequential definition, so sums are bit-identical to it; no atomics touch in_sum2.
#include "iq_common.cuh"

namespace iqk {

constexpr int kAccWarps = 8;          // warps per accumulate CTA
constexpr int kExpPerWarp = 16;       // experts a warp holds accumulators for (per expert batch)
constexpr int kExpBatch = kAccWarps * kExpPerWarp;  // 128 experts per pass over x
constexpr int kTileCols = 64;         // columns per accumulate CTA (2 per lane)

struct RouteWs {
  uint32_t *bits;      // [nchunks][E][W]
  int32_t *ccount;     // [nchunks][E]
  int32_t *order;      // [nchunks][E]
  int32_t *touched;    // [E]
};

__host__ __device__ inline size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

__host__ __device__ inline RouteWs route_ws(void *ws, int64_t nchunks, int E, int W) {
  uint8_t *p = (uint8_t *)ws;
  RouteWs r;
  r.bits = (uint32_t *)p; p += align256((size_t)nchunks * E * W * 4);
  r.ccount = (int32_t *)p; p += align256((size_t)nchunks * E * 4);
  r.order = (int32_t *)p; p += align256((size_t)nchunks * E * 4);
  r.touched = (int32_t *)p;
  return r;
}
static size_t route_ws_bytes(int64_t nchunks, int E, int W) {
  return align256((size_t)nchunks * E * W * 4) + 2 * align256((size_t)nchunks * E * 4) + align256((size_t)E * 4);
}

__global__ void __launch_bounds__(256) imatrix_route(const int32_t *__restrict__ ids, int64_t tokens, int top_k,
                                                     int E, int64_t rpc, int W, RouteWs ws,
                                                     unsigned long long *__restrict__ counts,
                                                     int32_t *__restrict__ status) {
  __shared__ int cnt[1024];
  const int64_t k = blockIdx.x;
  const int64_t t0 = k * rpc, t1 = min(tokens, t0 + rpc);
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  int st = 0;
  uint32_t *bits = ws.bits + (size_t)k * E * W;
  for (int64_t t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
    const int32_t *row = ids + t * top_k;
    const int r = (int)(t - t0);
    for (int a = 0; a < top_k; a++) {
      const int e = row[a];
      if (e < 0 || e >= E) { st |= IQ_STATUS_BAD_EXPERT_ID; continue; }
      bool dup = false;
      for (int b = 0; b < a; b++) dup |= (row[b] == e);
      if (dup) { st |= IQ_STATUS_DUP_EXPERT_ID; continue; }
      atomicOr(&bits[(size_t)e * W + (r >> 5)], 1u << (r & 31));
      atomicAdd(&cnt[e], 1);
    }
  }
  __syncthreads();
  // order experts by descending chunk count (ties: lower id first) with a rank count
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = cnt[e];
    int rank = 0;
    for (int o = 0; o < E; o++) {
      const int co = cnt[o];
      rank += (co > c) || (co == c && o < e);
    }
    ws.order[(size_t)k * E + rank] = e;
    ws.ccount[(size_t)k * E + e] = c;
    if (c) {
      atomicAdd(&counts[e], (unsigned long long)c);
      atomicOr(&ws.touched[e], 1);
    }
  }
  if (st && status) atomicOr(status, st);
}

template <typename T> struct AccIn;
template <> struct AccIn<__nv_bfloat16> { static constexpr int SUB = 256; using Pair = uint32_t; };
template <> struct AccIn<float> { static constexpr int SUB = 128; using Pair = uint64_t; };

// acc (a packed pair of fp32 partial sums) += (x0*x0, x1*x1): one rounded multiply and one rounded
// add per value (never fused), two values per instruction with the packed f32x2 forms.
__device__ __forceinline__ void sq_add(uint64_t &acc, uint64_t v) {
  uint64_t sq;
  asm("mul.rn.f32x2 %0, %1, %1;" : "=l"(sq) : "l"(v));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc) : "l"(sq));
}
__device__ __forceinline__ void sq_add(uint64_t &acc, uint32_t pr) {  // bf16 pair, widened exactly
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(pr << 16), "r"(pr & 0xffff0000u));
  sq_add(acc, v);
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kAccWarps * 32) imatrix_accumulate_kernel(
    const T *__restrict__ x, int64_t tokens, int64_t cols, int E, int64_t rpc, int W, RouteWs ws,
    float *__restrict__ in_sum2, int32_t *__restrict__ status) {
  constexpr int SUB = AccIn<T>::SUB;                 // rows per sub-tile
  constexpr int ROWB = kTileCols * (int)sizeof(T);   // bytes per sub-tile row
  constexpr int TILEB = SUB * ROWB;                  // bytes per sub-tile buffer
  using Pair = typename AccIn<T>::Pair;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *buf[2] = {smem, smem + TILEB};
  uint32_t *sbits = reinterpret_cast<uint32_t *>(smem + 2 * TILEB);  // [kExpBatch][SUB/32]

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t col0 = (int64_t)blockIdx.x * kTileCols;
  const int64_t nchunks = (tokens + rpc - 1) / rpc;
  const int subs_per_chunk = (int)((rpc + SUB - 1) / SUB);
  const int64_t nsteps = nchunks * subs_per_chunk;

  for (int eb = 0; eb < E; eb += kExpBatch) {
    const int ne = min(kExpBatch, E - eb);
    uint64_t acc[kExpPerWarp];  // packed (column 2*lane, column 2*lane+1) partial sums, +0.0f each
#pragma unroll
    for (int j = 0; j < kExpPerWarp; j++) acc[j] = 0ull;

    // issue the cp.async copies of sub-tile `step` into buffer step & 1
    auto issue = [&](int64_t step) {
      const int64_t k = step / subs_per_chunk;
      const int sidx = (int)(step % subs_per_chunk);
      const int64_t r0 = k * rpc + (int64_t)sidx * SUB;
      const int64_t r1 = min(min(tokens, (k + 1) * rpc), r0 + SUB);
      const int nrows = (int)(r1 - r0);
      uint8_t *dst = buf[step & 1];
      constexpr int PIECES = ROWB / 16;
      for (int i = threadIdx.x; i < nrows * PIECES; i += blockDim.x) {
        const int r = i / PIECES, c16 = i % PIECES;
        const uint8_t *src = reinterpret_cast<const uint8_t *>(x + (r0 + r) * cols + col0) + c16 * 16;
        cp_async16(dst + r * ROWB + c16 * 16, src);
      }
      cp_async_commit();
    };

    issue(0);
    for (int64_t step = 0; step < nsteps; step++) {
      const int64_t k = step / subs_per_chunk;
      const int sidx = (int)(step % subs_per_chunk);
      // stage this sub-tile's bitmap rows for the batch's experts
      const int wps = SUB / 32;
      for (int i = threadIdx.x; i < kExpBatch * wps; i += blockDim.x) {
        const int je = i / wps, wi = i % wps;
        const int gw = sidx * wps + wi;
        uint32_t v = 0;
        if (je < ne && gw < W) {
          const int e = ws.order[(size_t)k * E + eb + je];
          v = ws.bits[((size_t)k * E + e) * W + gw];
        }
        sbits[je * wps + wi] = v;
      }
      if (step + 1 < nsteps) { issue(step + 1); cp_async_wait<1>(); } else { cp_async_wait<0>(); }
      __syncthreads();
      const uint8_t *tile = buf[step & 1];
#pragma unroll
      for (int j = 0; j < kExpPerWarp; j++) {
        // snake deal over the count order: warp w takes positions w, 2*8-1-w, 16+w, ...
        const int je = j * kAccWarps + ((j & 1) ? (kAccWarps - 1 - warp) : warp);
        if (je >= ne) continue;
        for (int wi = 0; wi < wps; wi++) {
          uint32_t word = sbits[je * wps + wi];
          while (word) {
            const int r = wi * 32 + (__ffs(word) - 1);
            word &= word - 1;
            const Pair pr = reinterpret_cast<const Pair *>(tile + r * ROWB)[lane];
            sq_add(acc[j], pr);
          }
        }
      }
      __syncthreads();  // buffer step&1 is refilled two steps later; sbits is rewritten next step
      if (sidx == subs_per_chunk - 1) {
#pragma unroll
        for (int j = 0; j < kExpPerWarp; j++) {
          const int je = j * kAccWarps + ((j & 1) ? (kAccWarps - 1 - warp) : warp);
          if (je >= ne) continue;
          const int e = ws.order[(size_t)k * E + eb + je];
          if (ws.ccount[(size_t)k * E + e] == 0) continue;
          float2 *dst = reinterpret_cast<float2 *>(in_sum2 + (int64_t)e * cols + col0) + lane;
          float2 v = *dst;
          const float2 a = unpack2(acc[j]);
          v.x = __fadd_rn(v.x, a.x);
          v.y = __fadd_rn(v.y, a.y);
          *dst = v;
          acc[j] = 0ull;
        }
      }
    }
    // non-finite check of every expert this call touched (its rows of this column tile)
    if (status) {
      int bad = 0;
      for (int je = warp; je < ne; je += kAccWarps) {
        const int e = eb + je;
        if (!ws.touched[e]) continue;
        const float2 v = reinterpret_cast<const float2 *>(in_sum2 + (int64_t)e * cols + col0)[lane];
        bad |= !(isfinite(v.x) && isfinite(v.y));
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, IQ_STATUS_NONFINITE_SUM2);
    }
    __syncthreads();
  }
}

template <typename T>
static size_t acc_smem_bytes() {
  return 2 * (size_t)AccIn<T>::SUB * kTileCols * sizeof(T) + (size_t)kExpBatch * (AccIn<T>::SUB / 32) * 4;
}

}  // namespace iqk

using namespace iqk;

extern "C" int iq_imatrix_workspace_size(int64_t tokens, int num_experts, int64_t rows_per_chunk, size_t *bytes) {
  if (!bytes || tokens < 0 || num_experts <= 0 || num_experts > 1024 || rows_per_chunk <= 0 ||
      rows_per_chunk > 4096)
    return IQ_ERR_ARG;
  const int64_t nchunks = (tokens + rows_per_chunk - 1) / rows_per_chunk;
  const int W = (int)((rows_per_chunk + 31) / 32);
  *bytes = route_ws_bytes(nchunks, num_experts, W);
  return IQ_OK;
}

extern "C" int iq_imatrix_accumulate(const void *x, iq_dtype dt, int64_t tokens, int64_t cols,
                                     const int32_t *expert_ids, int top_k, int num_experts, int64_t rows_per_chunk,
                                     float *in_sum2, int64_t *counts, int32_t *status, void *workspace,
                                     size_t workspace_bytes, void *stream) {
  if (dt != IQ_F32 && dt != IQ_BF16) return IQ_ERR_ARG;
  if (tokens < 0 || cols <= 0 || cols % kTileCols || top_k < 1 || num_experts < top_k || num_experts > 1024 ||
      rows_per_chunk < 1 || rows_per_chunk > 4096)
    return IQ_ERR_ARG;
  if (!in_sum2 || !counts || (tokens > 0 && (!x || !expert_ids))) return IQ_ERR_ARG;
  if (((uintptr_t)x & 15) || ((uintptr_t)in_sum2 & 15) || ((uintptr_t)counts & 7) || ((uintptr_t)expert_ids & 3))
    return IQ_ERR_ARG;
  size_t need = 0;
  iq_imatrix_workspace_size(tokens, num_experts, rows_per_chunk, &need);
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255)) return IQ_ERR_WORKSPACE;
  if (tokens == 0) return IQ_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t nchunks = (tokens + rows_per_chunk - 1) / rows_per_chunk;
  const int W = (int)((rows_per_chunk + 31) / 32);
  RouteWs ws = route_ws(workspace, nchunks, num_experts, W);
  if (cudaMemsetAsync(workspace, 0, need, st) != cudaSuccess) return IQ_ERR_CUDA;
  imatrix_route<<<(unsigned)nchunks, 256, 0, st>>>(expert_ids, tokens, top_k, num_experts, rows_per_chunk, W, ws,
                                                   (unsigned long long *)counts, status);
  if (cudaPeekAtLastError() != cudaSuccess) return IQ_ERR_CUDA;
  const unsigned grid = (unsigned)(cols / kTileCols);
  if (dt == IQ_BF16) {
    const size_t sm = acc_smem_bytes<__nv_bfloat16>();
    cudaFuncSetAttribute(imatrix_accumulate_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    imatrix_accumulate_kernel<__nv_bfloat16><<<grid, kAccWarps * 32, sm, st>>>(
        (const __nv_bfloat16 *)x, tokens, cols, num_experts, rows_per_chunk, W, ws, in_sum2, status);
  } else {
    const size_t sm = acc_smem_bytes<float>();
    cudaFuncSetAttribute(imatrix_accumulate_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    imatrix_accumulate_kernel<float><<<grid, kAccWarps * 32, sm, st>>>(
        (const float *)x, tokens, cols, num_experts, rows_per_chunk, W, ws, in_sum2, status);
  }
  return cudaPeekAtLastError() == cudaSuccess ? IQ_OK : IQ_ERR_CUDA;
}

// ---------------------------------------------------------------------------------------------
namespace iqk {
__global__ void imatrix_weights_kernel(const float *__restrict__ s2, const int64_t *__restrict__ counts, int E,
                                       int64_t cols, float floor_, float *__restrict__ w) {
  const int64_t n = (int64_t)E * cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t c = counts[i / cols];
    if (c == 0) { w[i] = 1.0f; continue; }
    float m = __fdiv_rn(s2[i], __ll2float_rn(c));
    if (floor_ > 0.0f && m < floor_) m = floor_;
    w[i] = __fsqrt_rn(m);
  }
}
}  // namespace iqk

extern "C" int iq_imatrix_weights(const float *in_sum2, const int64_t *counts, int num_experts, int64_t cols,
                                  float floor, float *w, void *stream) {
  if (num_experts <= 0 || cols <= 0 || !in_sum2 || !counts || !w || w == in_sum2) return IQ_ERR_ARG;
  const int64_t n = (int64_t)num_experts * cols;
  const int64_t blocks = (n + 255) / 256;
  iqk::imatrix_weights_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, (cudaStream_t)stream>>>(
      in_sum2, counts, num_experts, cols, floor, w);
  return cudaPeekAtLastError() == cudaSuccess ? IQ_OK : IQ_ERR_CUDA;
}
