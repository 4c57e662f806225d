// Local-Hessian choice search (PR #3158 "local_hessian for GGML IQ", What does this PR do?) over
// the every-choice payloads (PR #3159 "one-pass every-choice encode").
//
// For a block (256 values of one row) and its dequantized values q_c under every choice c,
// dw_c = x - q_c.  H' = H_bb + perc_damp * mean(diag(H_bb)) * I is the damped 256 x 256 diagonal
// block of the input Hessian for the block's columns (damped as GPTQ damps).
//   Step 2: every group g takes argmin_c Q_g(c), Q_g(c) = dw_g(c)^T H'_gg dw_g(c) (lowest c on
//           equal values).
//   Step 3: two passes over the groups in ascending order; group g moves to the choice c that
//           minimises the block error dw^T H' dw with the other groups held, when that is strictly
//           lower than with its current choice (the lowest c among equal minima).  With
//           U = H'_{g, other groups} dw_{other groups} the change of the block error is
//               dE(c) = 2 (dw_g(c) - dw_g(cur)) . U_g + Q_g(c) - Q_g(cur),
//           so a visit costs one dot product of the group's width per choice, and a move updates
//           U by the product of the group's Hessian panel with the change of dw_g.
//
// Work layout: one CTA per (256-column block j, tile of kLhRows rows), 256 threads; thread i owns
// column i of the block in the U products.  The damped group-diagonal blocks of H', the tile's x,
// dw of the current choices, U and the Q_g(c) table live in shared memory; the off-diagonal panels
// of H' are read from global memory in coalesced rows (every tile of a column block reads the same
// 256 KB, which stays in L2).  The dequantized values of every choice are decoded on the fly from
// the payloads: per tile, each (row, choice) block's bytes are read once and unpacked in shared
// memory into the groups' local scales d (2s+1)[/8] and the vectors' (entry, signs or shift), and
// the codebook sits in shared memory, so a value costs a few shared-memory reads and one or two
// rounded products (the decoder's own arithmetic, so every value is the exact decoded one).  All
// arithmetic is fp32.
#include <cmath>

#include "iq_common.cuh"

namespace iqk {

constexpr int kLhRows = 16;      // rows per tile
constexpr int kLhThreads = 256;  // one thread per column of the block

template <int F> struct LhCfg {
  static constexpr int G = Fmt<F>::G, NC = Fmt<F>::C, GS = 256 / G, N = Fmt<F>::N;
  static constexpr int GPW = 32 / GS;  // groups a warp handles side by side (1 or 2)
  // Hgg [256][GS], Qe [kLhRows][G][NC], Xs / DWt / U [256][kLhRows], Dl [GS][kLhRows],
  // Ds [8 warps][32 lanes][NC], cur [kLhRows][G], codebook [N][8], local scales [kLhRows][NC][G],
  // vector codes [kLhRows][NC][32]
  static constexpr size_t SMEM = 4 * ((size_t)256 * GS + (size_t)kLhRows * G * NC + 3 * 256 * kLhRows +
                                      GS * kLhRows + 8 * 32 * NC + kLhRows * G + (size_t)N * 8 +
                                      (size_t)kLhRows * NC * G + (size_t)kLhRows * NC * 32) + 64;
  static_assert((size_t)kLhRows * NC * Fmt<F>::BB <= 2 * 256 * kLhRows * 4, "payload bytes fit the staging area");
};

// Unpacks one (row, choice) block from its payload bytes: the local scale of every group (IQ2
// d (2s+1) / 8, IQ1 d (2s+1), rounded as the decoder rounds them) and per vector its entry, its
// 8-bit sign mask (IQ2; bit 7 from even parity for IQ2_XXS / IQ2_XS) and its shift bit (IQ1).
template <int F>
__device__ __forceinline__ void lh_unpack(const uint8_t *pb, float *alph, uint32_t *code) {
  constexpr int G = Fmt<F>::G, VPG = Fmt<F>::VPG;
  uint32_t d16;
  if (F == IQ1_M) {
    d16 = 0;
#pragma unroll
    for (int k = 0; k < 4; k++) d16 |= get_bits(pb, f_d16_nib<F>(k)) << (4 * k);
  } else {
    d16 = get_bits(pb, f_d16<F>());
  }
  const float d = half_bits_to_float((uint16_t)d16);
  for (int g = 0; g < G; g++) {
    const int s = (int)get_bits(pb, f_scale<F>(g));
    alph[g] = Fmt<F>::IQ1 ? __fmul_rn(d, (float)(2 * s + 1)) : __fmul_rn(__fmul_rn(d, (float)(2 * s + 1)), 0.125f);
  }
  for (int v = 0; v < 32; v++) {
    const Bits lo = f_idx_lo<F>(v);
    const uint32_t idx = get_bits(pb, lo) | (get_bits(pb, f_idx_hi<F>(v)) << lo.width);
    uint32_t extra = 0;
    if (!Fmt<F>::IQ1) {
      uint32_t sg = get_bits(pb, f_sign<F>(v));
      if (Fmt<F>::PAR) sg |= (uint32_t)parity7((int)sg) << 7;
      extra = sg << 16;
    } else {
      const uint32_t db = F == IQ1_S ? get_bits(pb, f_dbit_grp<F>(v / VPG)) : get_bits(pb, f_dbit_vec<F>(v));
      extra = db << 24;
    }
    code[v] = idx | extra;
  }
}

// The decoded value of element i (0..255) of a block from its unpacked scales and codes.
template <int F>
__device__ __forceinline__ float lh_value(const float *alph, const uint32_t *code, const float *cbs, int i) {
  constexpr int GS = 256 / Fmt<F>::G;
  const uint32_t cd = code[i >> 3];
  const float gv = cbs[(cd & 0xffffu) * 8 + (i & 7)];
  const float al = alph[i / GS];
  if (!Fmt<F>::IQ1) {
    const float v = __fmul_rn(al, gv);
    return ((cd >> (16 + (i & 7))) & 1u) ? -v : v;
  }
  return __fmul_rn(al, __fadd_rn(gv, (cd >> 24) ? -0.125f : 0.125f));
}

// Packed fp32x2 multiply-add: two IEEE fp32 fma, each rounded on its own (the same values as two
// scalar __fmaf_rn).
__device__ __forceinline__ uint64_t lh_pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 lh_up2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t lh_fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// acc[4q .. 4q + 3] += h * d[q] for q < n4, as packed pairs
template <int n4>
__device__ __forceinline__ void lh_axpy4(uint64_t *acc2, float h, const float4 *d4) {
  const uint64_t hh = lh_pk2(h, h);
#pragma unroll
  for (int q = 0; q < n4; q++) {
    const float4 d = d4[q];
    acc2[2 * q] = lh_fma2(hh, lh_pk2(d.x, d.y), acc2[2 * q]);
    acc2[2 * q + 1] = lh_fma2(hh, lh_pk2(d.z, d.w), acc2[2 * q + 1]);
  }
}

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <int F, typename TIn>
__global__ void __launch_bounds__(kLhThreads, 1) lh_search_kernel(const TIn *__restrict__ W, int64_t rows, int64_t cols,
                                                               const uint8_t *__restrict__ payloads,
                                                               const float *__restrict__ grid,
                                                               const float *__restrict__ H, float perc_damp,
                                                               uint8_t *__restrict__ choices,
                                                               int32_t *__restrict__ status) {
  using Cfg = LhCfg<F>;
  constexpr int G = Cfg::G, NC = Cfg::NC, GS = Cfg::GS, GPW = Cfg::GPW, R = kLhRows, N = Cfg::N, BB = Fmt<F>::BB;
  extern __shared__ __align__(16) float sm[];
  float *Hgg = sm;                      // Hgg[(g*GS + b)*GS + a] = H'[g*GS + b][g*GS + a]
  float *Qe = Hgg + 256 * GS;           // [R][G][NC]
  float *Xs = Qe + R * G * NC;          // [256][R] x
  float *DWt = Xs + 256 * R;            // [256][R] dw of the current choices
  float *U = DWt + 256 * R;             // [256][R] off-diagonal products
  float *Dl = U + 256 * R;              // [GS][R] change of dw_g after a move
  float *Ds = Dl + GS * R;              // [8][32][NC] each warp's dw of every choice, for broadcast
  int *cur = reinterpret_cast<int *>(Ds + 8 * 32 * NC);  // [R][G]
  float *cbs = reinterpret_cast<float *>(cur + R * G);   // [N][8] codebook
  float *alph = cbs + N * 8;                              // [R][NC][G] local scales
  uint32_t *code = reinterpret_cast<uint32_t *>(alph + R * NC * G);  // [R][NC][32] vector codes
  uint8_t *pstage = reinterpret_cast<uint8_t *>(DWt);     // the tile's payload bytes (DWt and U, before use)
  // decoded value of element i of (row r, choice c) of the tile
  auto qv = [&](int r, int c, int i) { return lh_value<F>(alph + (r * NC + c) * G, code + (r * NC + c) * 32, cbs, i); };
  __shared__ float red[kLhThreads / 32];
  __shared__ int moved;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nb = cols / 256;
  const int64_t j = blockIdx.x;
  const float *Hj = H + (size_t)j * 256 * 256;
  const int64_t ntiles = (rows + R - 1) / R;
  for (int i = tid; i < N * 8; i += kLhThreads) cbs[i] = grid[i];

  // damping: lambda = perc_damp * mean(diag(H_bb))
  float dsum = Hj[(size_t)tid * 257];
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
  if (lane == 0) red[warp] = dsum;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < kLhThreads / 32; w++) tot += red[w];
  const float lam = perc_damp * (tot * (1.0f / 256.0f));
  if (!isfinite(lam)) {
    if (tid == 0 && blockIdx.y == 0 && status) atomicOr(status, IQ_STATUS_BAD_INPUT);
  }
  {  // damped group-diagonal blocks (column tid = g*GS + a)
    const int g = tid / GS, a = tid % GS;
    for (int b = 0; b < GS; b++) {
      const float h = Hj[(size_t)(g * GS + b) * 256 + g * GS + a];
      Hgg[(g * GS + b) * GS + a] = b == a ? __fadd_rn(h, lam) : h;
    }
  }
  __syncthreads();

  for (int64_t tile = blockIdx.y; tile < ntiles; tile += gridDim.y) {
    const int64_t r0 = tile * R;
    const int nr = (int)min((int64_t)R, rows - r0);
    // ---- x of the tile ---------------------------------------------------------------------
    for (int r = 0; r < R; r++)
      Xs[tid * R + r] = r < nr ? to_f(W[(size_t)(r0 + r) * cols + j * 256 + tid]) : 0.0f;
    // ---- every (row, choice) block of the tile: bytes staged, then unpacked --------------------
    static_assert(BB % 2 == 0, "payload blocks are whole 16-bit words");
    for (int t = tid; t < R * NC * (BB / 2); t += kLhThreads) {   // 16-bit words (blocks start even)
      const int rc = t / (BB / 2), bi = t % (BB / 2), r = rc / NC, c = rc % NC;
      reinterpret_cast<uint16_t *>(pstage)[t] =
          r < nr ? reinterpret_cast<const uint16_t *>(payloads + ((size_t)c * rows * nb + (size_t)(r0 + r) * nb + j) * BB)[bi]
                 : (uint16_t)0;
    }
    __syncthreads();
    if (tid < R * NC) lh_unpack<F>(pstage + tid * BB, alph + tid * G, code + tid * 32);
    __syncthreads();
    // ---- step 2: Q_g(c) for every (row, group, choice) -------------------------------------
    for (int u = warp; u < R * (G / GPW); u += kLhThreads / 32) {
      const int r = u / (G / GPW);
      const int g = (u % (G / GPW)) * GPW + lane / GS, a = lane % GS;
      const int i = g * GS + a;
      if (r < nr) {
        // every choice side by side: NC independent multiply-add chains over the group
        const float x = Xs[i * R + r];
        float dw[NC];
        uint64_t y2[NC / 2];
        float *ds = Ds + warp * 32 * NC;  // lane's row: the NC values of its element
#pragma unroll
        for (int c = 0; c < NC; c++) dw[c] = __fsub_rn(x, qv(r, c, i));
#pragma unroll
        for (int c = 0; c < NC / 2; c++) y2[c] = 0ull;
#pragma unroll
        for (int c = 0; c < NC; c += 4)
          *reinterpret_cast<float4 *>(ds + lane * NC + c) = make_float4(dw[c], dw[c + 1], dw[c + 2], dw[c + 3]);
        __syncwarp();
        const float *seg = ds + (lane / GS) * GS * NC;  // the lane's group's elements
#pragma unroll 2
        for (int b = 0; b < GS; b++)
          lh_axpy4<NC / 4>(y2, Hgg[(g * GS + b) * GS + a], reinterpret_cast<const float4 *>(seg + b * NC));
        __syncwarp();
#pragma unroll
        for (int c = 0; c < NC; c++) {
          const float2 yp = lh_up2(y2[c / 2]);
          float p = __fmul_rn(dw[c], (c & 1) ? yp.y : yp.x);
#pragma unroll
          for (int off = GS / 2; off >= 1; off >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, off, GS));
          if (a == 0) Qe[(r * G + g) * NC + c] = p;
        }
      }
    }
    __syncthreads();
    if (tid < R * G) {
      const int r = tid / G, g = tid % G;
      const float *q = Qe + (r * G + g) * NC;
      float best = q[0];
      int bc = 0;
      for (int c = 1; c < NC; c++)
        if (q[c] < best) { best = q[c]; bc = c; }
      cur[r * G + g] = bc;
    }
    __syncthreads();
    {  // dw of the current choices
      const int g = tid / GS;
      for (int r = 0; r < R; r++)
        DWt[tid * R + r] = r < nr ? __fsub_rn(Xs[tid * R + r], qv(r, cur[r * G + g], tid)) : 0.0f;
    }
    __syncthreads();
    // ---- U = H'_offdiag dw: thread tid owns column tid (in registers; the visited group's slice is
    // published to shared memory before each visit) ----------------------------------------------
    uint64_t ureg2[R / 2];   // U of this thread's column for the tile's rows, as packed pairs
    {
      const int gi = tid / GS;
#pragma unroll
      for (int r = 0; r < R / 2; r++) ureg2[r] = 0ull;
      for (int kg = 0; kg < G; kg++) {
        if (kg == gi) continue;
#pragma unroll 16
        for (int kk = 0; kk < GS; kk++) {
          const int k = kg * GS + kk;
          lh_axpy4<R / 4>(ureg2, __ldg(Hj + (size_t)k * 256 + tid), reinterpret_cast<const float4 *>(DWt + k * R));
        }
      }
    }
    // ---- step 3: two revisits ------------------------------------------------------------------
    for (int pass = 0; pass < 2; pass++) {
      for (int g = 0; g < G; g++) {
        // group g's Hessian panel for this thread's column, loaded now so its latency overlaps the
        // move evaluation (used only if a row moves)
        float hp[GS];
        if (tid / GS != g) {
#pragma unroll
          for (int k = 0; k < GS; k++) hp[k] = __ldg(Hj + (size_t)(g * GS + k) * 256 + tid);
        }
        if (tid == 0) moved = 0;
        if (tid / GS == g) {
#pragma unroll
          for (int r = 0; r < R / 2; r++) {
            const float2 u2 = lh_up2(ureg2[r]);
            U[tid * R + 2 * r] = u2.x;
            U[tid * R + 2 * r + 1] = u2.y;
          }
        }
        __syncthreads();
        // (a) every row's best move for group g: a warp per row, GPW choices side by side
        for (int r = warp; r < R; r += kLhThreads / 32) {
          const int a = lane % GS, i = g * GS + a;
          const int cc = r < nr ? cur[r * G + g] : 0;
          float bestd = 0.0f;
          int bestc = cc;
          if (r < nr) {
            const float x = Xs[i * R + r], dcur = DWt[i * R + r], uu = U[i * R + r];
            const float qcur = Qe[(r * G + g) * NC + cc];
            constexpr int NS = NC / GPW;  // steps; step s holds choices s * GPW + (lane / GS)
            float t[NS];
#pragma unroll
            for (int st = 0; st < NS; st++) {
              const int c = st * GPW + lane / GS;
              const float dwc = __fsub_rn(x, qv(r, c, i));
              t[st] = __fmul_rn(__fsub_rn(dwc, dcur), uu);
            }
#pragma unroll
            for (int off = GS / 2; off >= 1; off >>= 1)
#pragma unroll
              for (int st = 0; st < NS; st++) t[st] = __fadd_rn(t[st], __shfl_xor_sync(0xffffffffu, t[st], off, GS));
            // choices in ascending order: segment 0 holds the step's first choice, segment 1 (GPW = 2)
            // the next one
#pragma unroll
            for (int st = 0; st < NS; st++) {
              const int c = st * GPW + lane / GS;
              const float dE = __fadd_rn(__fmul_rn(2.0f, t[st]), __fsub_rn(Qe[(r * G + g) * NC + c], qcur));
#pragma unroll
              for (int s = 0; s < GPW; s++) {
                const float v = __shfl_sync(0xffffffffu, dE, s * GS);
                if (v < bestd) { bestd = v; bestc = st * GPW + s; }
              }
            }
          }
          // (b) apply the move: new dw_g, its change, the choice
          if (r < nr && bestc != cc) {
            if (lane < GS) {
              const float x = Xs[i * R + r];
              const float dwn = __fsub_rn(x, qv(r, bestc, i));
              Dl[a * R + r] = __fsub_rn(dwn, DWt[i * R + r]);
              DWt[i * R + r] = dwn;
            }
            if (lane == 0) { cur[r * G + g] = bestc; moved = 1; }
          } else if (lane < GS) {
            Dl[a * R + r] = 0.0f;
          }
        }
        __syncthreads();
        // (c) U of the other groups' columns += H'[., g panel] * change
        if (moved && tid / GS != g) {
#pragma unroll
          for (int k = 0; k < GS; k++) lh_axpy4<R / 4>(ureg2, hp[k], reinterpret_cast<const float4 *>(Dl + k * R));
        }
        __syncthreads();
      }
    }
    // ---- the tile's choices ------------------------------------------------------------------
    if (tid < R * G) {
      const int r = tid / G, g = tid % G;
      if (r < nr) choices[((size_t)(r0 + r) * nb + j) * G + g] = (uint8_t)cur[r * G + g];
    }
    __syncthreads();
  }
}

template <int F, typename TIn>
static int run_lh(const void *W, int64_t rows, int64_t cols, const uint8_t *payloads, const float *grid,
                  const float *H, float perc_damp, uint8_t *choices, int32_t *status, cudaStream_t st) {
  const size_t smem = LhCfg<F>::SMEM;
  auto kern = lh_search_kernel<F, TIn>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return IQ_ERR_CUDA;
  const int64_t ntiles = (rows + kLhRows - 1) / kLhRows;
  const dim3 grid_dim((unsigned)(cols / 256), (unsigned)(ntiles < 65535 ? ntiles : 65535));
  kern<<<grid_dim, kLhThreads, smem, st>>>((const TIn *)W, rows, cols, payloads, grid, H, perc_damp, choices, status);
  return cudaPeekAtLastError() == cudaSuccess ? IQ_OK : IQ_ERR_CUDA;
}

}  // namespace iqk

using namespace iqk;

static int lh_num_choices(iq_format f) { return f == IQ1_M ? 8 : 16; }

extern "C" int iq_local_hessian_workspace_size(iq_format f, int64_t rows, int64_t cols, size_t *bytes) {
  if ((unsigned)f > IQ1_M || rows < 0 || cols <= 0 || cols % 256 || !bytes) return IQ_ERR_ARG;
  *bytes = 0;  // the search decodes the payloads itself and needs no scratch
  return IQ_OK;
}

extern "C" int iq_local_hessian_choices(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols,
                                        const float *grid, const uint8_t *payloads, const float *hessian,
                                        float perc_damp, uint8_t *choices, int32_t *status, void *workspace,
                                        size_t workspace_bytes, void *stream) {
  if ((unsigned)f > IQ1_M || (dt != IQ_F32 && dt != IQ_BF16) || rows < 0 || cols <= 0 || cols % 256)
    return IQ_ERR_ARG;
  if (cols / 256 > 65535) return IQ_ERR_ARG;
  if (!(perc_damp >= 0.0f) || !std::isfinite(perc_damp)) return IQ_ERR_ARG;
  const int64_t nb = rows * (cols / 256);
  if (nb == 0) return IQ_OK;
  if (!W || !grid || !payloads || !hessian || !choices) return IQ_ERR_ARG;
  if (((uintptr_t)W & 15) || ((uintptr_t)grid & 15) || ((uintptr_t)hessian & 15) || ((uintptr_t)payloads & 1))
    return IQ_ERR_ARG;
  (void)workspace;
  (void)workspace_bytes;
  cudaStream_t st = (cudaStream_t)stream;
  switch (f) {
#define LH_CASE(FMT)                                                                                      \
  case FMT:                                                                                               \
    return dt == IQ_BF16                                                                                 \
               ? run_lh<FMT, __nv_bfloat16>(W, rows, cols, payloads, grid, hessian, perc_damp, choices, status, st) \
               : run_lh<FMT, float>(W, rows, cols, payloads, grid, hessian, perc_damp, choices, status, st);
    LH_CASE(IQ2_XXS)
    LH_CASE(IQ2_XS)
    LH_CASE(IQ2_S)
    LH_CASE(IQ1_S)
    LH_CASE(IQ1_M)
#undef LH_CASE
  }
  return IQ_ERR_ARG;
}
