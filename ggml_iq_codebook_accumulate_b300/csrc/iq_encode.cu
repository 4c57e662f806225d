// Importance-weighted codebook encoder for the GGML IQ formats, its every-choice error table and
// the super-block anchor.
//
// Sources: PR #2513 (IQ2_XXS / IQ2_S / IQ1_M commit texts: single-pass grid search at a fixed
// anchored super-block scale, even-parity sign rule, full sign mask for IQ2_S, +-1/8 shift for IQ1,
// tie order (lower shift, then lower entry), anchors); PR #3157 "[1/5] Let the GGML IQ encoders take
// fixed per-group choices" (one choice per group by least weighted squared error, fixed choices keep
// the entry search, choices in [0, num_choices), zero blocks); PR #3159 (every choice from one
// sweep).
//
// Work layout: one warp per 256-value block, lane g = vector g (8 values).  The codebook, prepared
// as [entry][g(8) | g^2 or |g| (8)] fp32, is copied once per CTA into dynamic shared memory with a
// bulk async copy (TMA engine, mbarrier completion) and read as warp-wide broadcasts.
//
// For vector v with weights w, targets t (signed magnitudes for IQ2, x for IQ1) and a candidate
// (entry e [, shift delta]) under local scale alpha, the error is
//     E = sum w (t - alpha u)^2 = Cs + alpha * s,   s = alpha * B - 2 A,
// with u = g (IQ2) or g + delta (IQ1), A = sum w t u, B = sum w u^2, Cs = sum w t^2.  The sweep
// computes A and B once per entry (FMA chains) and s for every choice (one FMA + one min each), so
// per (vector, choice) it keeps min_e s.  The group's choice minimises alpha * sum_v min s; the
// vector's candidate under that choice is found by a second sweep at one alpha.
//
// Exactness: every decision the fp32 sweep makes with a gap larger than its rounding bound
// (kMargin, see iq_common.cuh) equals the exact decision.  Smaller gaps are flagged per block; a
// second kernel rescores the flagged groups: it screens candidates in fp32 and evaluates every
// candidate the bound cannot exclude with the direct fp64 form sum_i w_i (x_i - q_i)^2 of the
// decoded values q, then takes the exact minimum with the lowest (choice) / (delta bit, entry) on
// equal error.
#include <mutex>
#include <type_traits>

#include "iq_common.cuh"

namespace iqk {

// searched (+ every-choice table), fixed choices, every-choice table only, every-choice payloads
enum { MODE_SEARCH = 0, MODE_FIXED = 1, MODE_TABLE = 2, MODE_EVERY = 3 };

__host__ __device__ inline size_t al256(size_t n) { return (n + 255) & ~(size_t)255; }

struct EncWs {
  int32_t *hdr;  // [0] codebook invalid, [1] number of flagged blocks, [2] rescoring's next item
  float4 *tab;   // [N][4] prepared codebook
  uint2 *fb;     // [B] flagged blocks: (block index, vector mask)
};
__host__ __device__ inline EncWs enc_ws(void *ws, int N) {
  uint8_t *p = (uint8_t *)ws;
  EncWs r;
  r.hdr = (int32_t *)p; p += 256;
  r.tab = (float4 *)p; p += al256((size_t)N * 64);
  r.fb = (uint2 *)p;
  return r;
}
static size_t enc_ws_bytes(int N, int64_t nblocks) { return 256 + al256((size_t)N * 64) + al256((size_t)nblocks * 8); }

struct EncArgs {
  const void *W;
  int64_t rows, cols, nblocks;
  const float *imp;
  int64_t rows_per_expert;
  const float *grid;
  const uint16_t *d16;
  const uint8_t *choices;  // fixed mode: [B][G], or null with every group at uniform_choice
  uint8_t *payload;
  float *table;
  int32_t *status;
  int uniform_choice;
  void *wb;  // write-back: W (same dtype) overwritten with the decoded payload, or null
};

// the fixed choice of group g of block b
template <int G> __device__ __forceinline__ int fixed_choice(const EncArgs &a, int64_t b, int g) {
  return a.choices ? (int)a.choices[b * G + g] : a.uniform_choice;
}

// Write-back of one vector (lane `lane` of block b): its 8 decoded values by the value rule
// (IQ2 q = d (2s+1)/8 g, negated where sign bit i is set; IQ1 q = d (2s+1) (g + delta)), stored in
// W's dtype (fp32 exact: every decoded value is an exact fp32 product; bf16 rounded to nearest
// even).  g8: the entry's 8 codebook values.  Zero scale or a rejected block: d = 0 gives zeros.
__device__ __forceinline__ void store8(float *o, const float *q) {
  reinterpret_cast<float4 *>(o)[0] = make_float4(q[0], q[1], q[2], q[3]);
  reinterpret_cast<float4 *>(o)[1] = make_float4(q[4], q[5], q[6], q[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16 *o, const float *q) {
  uint32_t u[4];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(q[2 * k], q[2 * k + 1]);
    u[k] = *reinterpret_cast<const uint32_t *>(&h2);
  }
  *reinterpret_cast<uint4 *>(o) = make_uint4(u[0], u[1], u[2], u[3]);
}
template <int F, typename TIn>
__device__ __forceinline__ void write_back_vec(const EncArgs &a, int64_t b, int lane, const float *g8, float d, int s,
                                               int sgn, int dbit) {
  float q[8];
  if (!Fmt<F>::IQ1) {
    const float dl = __fmul_rn(__fmul_rn(d, (float)(2 * s + 1)), 0.125f);
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const float v = __fmul_rn(dl, g8[i]);
      q[i] = ((sgn >> i) & 1) ? -v : v;
    }
  } else {
    const float dl = __fmul_rn(d, (float)(2 * s + 1));
    const float delta = dbit ? -0.125f : 0.125f;
#pragma unroll
    for (int i = 0; i < 8; i++) q[i] = __fmul_rn(dl, __fadd_rn(g8[i], delta));
  }
  const int64_t bpr = a.cols / 256;
  TIn *W = reinterpret_cast<TIn *>(a.wb);
  store8(W + (b / bpr) * a.cols + (b % bpr) * 256 + lane * 8, q);
}
// Write-back of a rejected or zero-scale block: the decode of its all-zero payload (scale 0, entry
// 0, choice 0, no signs, delta bit 0), whose values are zeros carrying the sign of entry 0's
// values (+- 0 for IQ1, where g + delta can be negative).
template <int F, typename TIn>
__device__ __forceinline__ void write_back_zero(const EncArgs &a, int64_t b, int lane) {
  float g8[8];
  load8(a.grid, g8);
  write_back_vec<F, TIn>(a, b, lane, g8, 0.0f, 0, 0, 0);
}

// ---------------------------------------------------------------------------------------------
// Prepared codebook: g [N x 8] then h [N x 8] (h = g^2 for IQ2, |g| for IQ1), each a K-major
// operand of the tensor-core sweep in the canonical no-swizzle layout (see kmaj below).
__host__ __device__ __forceinline__ int kmaj(int row, int k) {
  return (row >> 3) * 64 + (k >> 2) * 32 + (row & 7) * 4 + (k & 3);
}

template <int F>
__global__ void prep_codebook(const float *__restrict__ grid, EncWs ws) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= Fmt<F>::N) return;
  float g[8];
  load8(grid + 8 * e, g);
  bool ok = true;
  float *tf = reinterpret_cast<float *>(ws.tab);
#pragma unroll
  for (int i = 0; i < 8; i++) {
    float h;
    if (Fmt<F>::IQ1) {
      ok &= (g[i] == -1.0f || g[i] == 0.0f || g[i] == 1.0f);
      h = fabsf(g[i]);
    } else {
      ok &= (g[i] >= 1.0f && g[i] <= 127.0f && g[i] == floorf(g[i]));
      h = g[i] * g[i];  // exact: at most 14 bits
    }
    tf[kmaj(e, i)] = g[i];
    tf[Fmt<F>::N * 8 + kmaj(e, i)] = h;
  }
  if (!ok) atomicOr(&ws.hdr[0], 1);
}

struct Entry { float g[8], h[8]; };
// Entry e from the caller's codebook [N][8] (two 16-byte loads), with h formed as prep_codebook
// forms it (g^2 for IQ2, |g| for IQ1; exact).
template <int F>
__device__ __forceinline__ void load_entry(const float *grid, int e, Entry &en) {
  const float4 p = __ldg(reinterpret_cast<const float4 *>(grid + 8 * e));
  const float4 q = __ldg(reinterpret_cast<const float4 *>(grid + 8 * e) + 1);
  en.g[0] = p.x; en.g[1] = p.y; en.g[2] = p.z; en.g[3] = p.w;
  en.g[4] = q.x; en.g[5] = q.y; en.g[6] = q.z; en.g[7] = q.w;
#pragma unroll
  for (int i = 0; i < 8; i++) en.h[i] = Fmt<F>::IQ1 ? fabsf(en.g[i]) : __fmul_rn(en.g[i], en.g[i]);
}

// ---------------------------------------------------------------------------------------------
// Packed f32x2 arithmetic (two IEEE fp32 operations per instruction, each rounded on its own).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 up2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ---------------------------------------------------------------------------------------------
// Per-vector state.
struct Vec {
  float x[8], w[8];
  float nw2[8];  // -2 * w * t (exact scaling of the rounded product w*t)
  float Cs;      // sum w t^2 (fp32, only for the rounding bound)
  float nT2;     // sum of nw2 (IQ1)
  float Ws;      // sum of w (IQ1)
  int sgn;       // IQ2 sign mask
};

template <int F>
__device__ __forceinline__ void vec_setup(Vec &v) {
  float t[8];
  if (!Fmt<F>::IQ1) {
    v.sgn = sign_rule<F>(v.x, v.w, t);
  } else {
    v.sgn = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) t[i] = v.x[i];
  }
  float cs = 0.0f, nt = 0.0f, ws = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const float wt = __fmul_rn(v.w[i], t[i]);
    v.nw2[i] = -2.0f * wt;
    cs = __fmaf_rn(wt, t[i], cs);
    nt = __fadd_rn(nt, v.nw2[i]);
    ws = __fadd_rn(ws, v.w[i]);
  }
  v.Cs = cs; v.nT2 = nt; v.Ws = ws;
}

// The per-entry sums, scalar (rescoring) and packed over an entry pair (sweeps).  Both evaluate
// the same rounded operations in the same order, so their fp32 values agree bit for bit:
//   An = -2 sum w t g   (first product rounded, then a chain of FMAs over i = 1..7)
//   B  = sum w h        (IQ2: h = g^2, IQ1: h = |g| = g^2)
//   Cg = sum w g        (IQ1)
// and for IQ1 the sums of the shifted values g + delta, delta = +-1/8:
//   Anp/Anm = An +- nT2/8,   Bp/Bm = (B + Ws/64) +- Cg/4.
__device__ __forceinline__ void ab2(const float *nw2, const float *w, const Entry &en, float &An, float &B) {
  An = __fmul_rn(nw2[0], en.g[0]);
  B = __fmul_rn(w[0], en.h[0]);
#pragma unroll
  for (int i = 1; i < 8; i++) { An = __fmaf_rn(nw2[i], en.g[i], An); B = __fmaf_rn(w[i], en.h[i], B); }
}
__device__ __forceinline__ void ab1(const Vec &v, const Entry &en, float &Anp, float &Bp, float &Anm, float &Bm) {
  float An = __fmul_rn(v.nw2[0], en.g[0]), Cg = __fmul_rn(v.w[0], en.g[0]), B = __fmul_rn(v.w[0], en.h[0]);
#pragma unroll
  for (int i = 1; i < 8; i++) {
    An = __fmaf_rn(v.nw2[i], en.g[i], An);
    Cg = __fmaf_rn(v.w[i], en.g[i], Cg);
    B = __fmaf_rn(v.w[i], en.h[i], B);
  }
  Anp = __fmaf_rn(0.125f, v.nT2, An);
  Anm = __fmaf_rn(-0.125f, v.nT2, An);
  const float Bw = __fmaf_rn(0.015625f, v.Ws, B);
  Bp = __fmaf_rn(0.25f, Cg, Bw);
  Bm = __fmaf_rn(-0.25f, Cg, Bw);
}

struct IQ1Const { uint64_t p125, m125, p025, m025, w64; };
__device__ __forceinline__ IQ1Const iq1_consts() {
  return {pk2(0.125f, 0.125f), pk2(-0.125f, -0.125f), pk2(0.25f, 0.25f), pk2(-0.25f, -0.25f),
          pk2(0.015625f, 0.015625f)};
}

// local scale multipliers: IQ2 alpha_s = d * (2s+1) / 8, IQ1 alpha_s = d * (2s+1) (both exact)
template <int F> __device__ __forceinline__ float alpha_of(float d, int s) {
  return Fmt<F>::IQ1 ? __fmul_rn(d, (float)(2 * s + 1)) : __fmul_rn(__fmul_rn(d, (float)(2 * s + 1)), 0.125f);
}
// alpha of choice c (IQ1_S: scale = c & 7)
template <int F> __device__ __forceinline__ float alpha_choice(float d, int c) {
  return alpha_of<F>(d, F == IQ1_S ? (c & 7) : c);
}

// best / runner-up / key over a pair of candidates (keys ka and ka + 1)
__device__ __forceinline__ void track2(float2 sc, int ka, float &best, float &second, int &key) {
  const float lo = fminf(sc.x, sc.y), hi = fmaxf(sc.x, sc.y);
  const int klo = sc.y < sc.x ? ka + 1 : ka;
  second = min3f(second, hi, fmaxf(best, lo));
  if (lo < best) { best = lo; key = klo; }
}

// ---------------------------------------------------------------------------------------------
// Copy the prepared codebook (bytes, multiple of 16) into shared memory with bulk async copies;
// every thread waits on the mbarrier for at most ~2 s.  Returns false on timeout.
__device__ bool load_codebook(float4 *dst, const float4 *src, uint32_t bytes, uint64_t *mbar) {
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(mbar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(mbar)), "r"(bytes)
                 : "memory");
    constexpr uint32_t CH = 32768;
    for (uint32_t off = 0; off < bytes; off += CH) {
      const uint32_t n = bytes - off < CH ? bytes - off : CH;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              smem_u32(reinterpret_cast<uint8_t *>(dst) + off)),
          "l"(reinterpret_cast<const uint8_t *>(src) + off), "r"(n), "r"(smem_u32(mbar))
          : "memory");
    }
  }
  const uint64_t t0 = global_timer_ns();
  bool done = false;
  while (!done) {
    done = mbar_try_wait(mbar, 0);
    if (!done && global_timer_ns() - t0 > 2000000000ull) break;
  }
  return done;
}

template <typename TIn>
__device__ __forceinline__ void load_block_vec(const EncArgs &a, int64_t b, int lane, Vec &v) {
  const int64_t bpr = a.cols / 256;
  const int64_t row = b / bpr, kb = b % bpr;
  const TIn *W = reinterpret_cast<const TIn *>(a.W);
  load8(W + row * a.cols + kb * 256 + lane * 8, v.x);
  if (a.imp) {
    const int64_t er = a.rows_per_expert > 0 ? row / a.rows_per_expert : 0;
    load8(a.imp + er * a.cols + kb * 256 + lane * 8, v.w);
  } else {
#pragma unroll
    for (int i = 0; i < 8; i++) v.w[i] = 1.0f;
  }
}

// Validates the block and returns its scale bits; 0 means "write an all-zero payload".  d16in: the
// given scale bits of the block (read ahead), or -1 to compute the anchor; cin: lane g < G holds the
// fixed choice of group g (read ahead; fixed-choice mode).
template <int F, int MODE>
__device__ __forceinline__ uint32_t block_scale(const Vec &v, int lane, int d16in, int cin, int &bad_bits) {
  constexpr int G = Fmt<F>::G, C = Fmt<F>::C;
  bad_bits = 0;
  bool fin = finite8(v.x);
  bool wok = true;
#pragma unroll
  for (int i = 0; i < 8; i++) wok &= (v.w[i] >= 0.0f) && isfinite(v.w[i]);
  if (!__all_sync(0xffffffffu, fin)) bad_bits |= IQ_STATUS_BAD_INPUT;
  else if (!__all_sync(0xffffffffu, wok)) bad_bits |= IQ_STATUS_BAD_IMPORTANCE;
  if (bad_bits) return 0;
  uint32_t d16 = d16in >= 0 ? (uint32_t)d16in : (uint32_t)half_bits_rn(anchor_scale<F>(v.x));
  if ((d16 & 0x7c00u) == 0x7c00u || ((d16 & 0x8000u) && (d16 & 0x7fffu))) { bad_bits |= IQ_STATUS_BAD_SCALE; return 0; }
  d16 &= 0x7fffu;
  if (MODE == MODE_FIXED) {
    if (__any_sync(0xffffffffu, lane < G && cin >= C)) { bad_bits |= IQ_STATUS_BAD_CHOICE; return 0; }
  }
  return d16;
}

// Group reduction over the VPG lanes of each choice group, in vector order.
template <int VPG>
__device__ __forceinline__ float group_sum(float val, int g0) {
  float s = __shfl_sync(0xffffffffu, val, g0);
#pragma unroll
  for (int k = 1; k < VPG; k++) s = __fadd_rn(s, __shfl_sync(0xffffffffu, val, g0 + k));
  return s;
}

// ---------------------------------------------------------------------------------------------
// Tensor-core sweep.
//
// A CTA encodes 4 blocks (128 vectors) at a time.  The per-entry sums of every vector are the
// product of a [128 x 8] per-vector operand and the [8 x N] codebook:
//     An = -2 (w t) . g        B = w . h (h = g^2 or |g|)        Cg = w . g (IQ1)
// evaluated by tcgen05.mma (kind::tf32, fp32 accumulators in tensor memory), 64 codebook entries
// per chunk.  The codebook values g (integers of at most 7 bits) are exact in tf32; h = g^2 of
// an IQ2 grid can need 14 bits, so it is split into exact tf32 parts hi + lo when any entry needs
// it (two more MMAs for B).  Each fp32 per-vector operand is split into two tf32 parts (hi, lo =
// x - hi, each rounded to tf32) accumulated into the same tensor-memory column: every product of
// a part is exact, the split leaves at most 2^-22 of each operand, and the sums carry the
// accumulation rounding (together measured on B300 at most 6.3 units of 2^-24 of sum |a*b|,
// inside the same rounding margin as an fp32 FMA chain).
// A control warp issues the MMAs into a double-buffered tensor-memory region and commits each
// chunk to an mbarrier; 8 consumer warps (2 per tensor-memory lane quarter = block) load their 32
// columns per chunk with tcgen05.ld and do the per-choice scoring with packed f32x2 FMAs and
// three-input minima, then release the buffer.  Sweep 1 keeps, per vector and choice, the minimum
// score; sweep 2 (same MMAs) finds each vector's best candidate and runner-up under the chosen
// choice.  All waits are bounded.

// kmaj(row, k): float offset of (row, k) in a K-major [rows x 8] fp32 operand in the canonical
// no-swizzle layout: 8-row x 16-byte core matrices of 128 contiguous bytes, K-adjacent core
// matrices 128 bytes apart (leading byte offset), row-group-adjacent ones 256 bytes apart (stride
// byte offset).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(256 >> 4) << 32) |
         (1ull << 46);
}
// instruction descriptor: D fp32, A and B tf32, both K-major, M = 128, N = NN
template <int NN> __host__ __device__ constexpr uint32_t umma_idesc() {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(NN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void umma_tf32(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(mbar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// merges a second tracker (b2, s2, k2) into (best, second, key): the lower score wins, the lower
// key on equal scores
__device__ __forceinline__ void merge_track(float &best, float &second, int &key, float b2, float s2, int k2) {
  const bool take = b2 < best || (b2 == best && k2 < key);
  second = min3f(second, s2, fmaxf(best, b2));
  if (take) { best = b2; key = k2; }
}

// 16 consecutive fp32 columns of the warp's 32 tensor-memory lanes (thread t: lane base + t)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

constexpr int kTcConsumers = 8;                      // 2 consumer warps per block of the quad
constexpr int kCtrlWarp = kTcConsumers;              // issues the MMAs
constexpr int kPrepWarp = kTcConsumers + 1;          // first of the warps preparing the next quad
constexpr int kPrepWarps = 2;                        // each prepares 2 of the quad's 4 blocks
constexpr int kTcThreads = (kTcConsumers + 1 + kPrepWarps) * 32;
constexpr int kChunk = 64;                           // codebook entries per MMA chunk
constexpr size_t kMaxDynSmem = 227 * 1024;

template <int F> struct TcCfg {
  static constexpr int NQ = Fmt<F>::IQ1 ? 3 : 2;       // An, (Cg), B columns per entry
  static constexpr int NCH = Fmt<F>::N / kChunk;        // chunks per sweep
  static constexpr int ALLOC = 2 * NQ * kChunk <= 256 ? 256 : 512;  // tensor-memory columns
  // IQ2: h = g^2 may need more significant bits than tf32 holds; its low part goes here
  static constexpr size_t HLO = Fmt<F>::IQ1 ? 0 : (size_t)Fmt<F>::N * 32;
  // shared memory besides the per-vector operands (tc_na below, 4 KB each)
  static constexpr size_t SMEM = (size_t)Fmt<F>::N * 64 + HLO + 2 * 128 * 16 * 4 + 2 * 128 * 4 * 4 + 4 * 24 * 4;
  // every-choice payloads: per (warp half, vector, choice) the minimum, the near bound (fp32) and
  // key | count << 16
  static constexpr size_t EVERY = 2 * 128 * 16 * 4 * 3;
  // per-quad state from the prep warp: per vector (Cs, nT2, Ws, sign mask), per block d16 | active
  static constexpr size_t STATE = 128 * 16 + 4 * 4;
};

// Per-vector [128 x 8] tf32 operands: nw2 hi, nw2 lo, w hi, w lo; for the second sweep of the
// searched and fixed modes, IQ1_M: w/4 hi, w/4 lo, -w/4 hi, -w/4 lo; IQ1_S: sigma w/4 hi,
// sigma w/4 lo with sigma = +-1 the sign of the group's shift, given (fixed choices) or chosen by
// the first sweep (written between the sweeps) (the shifted sums' MMAs, below).
template <int F, int MODE> __host__ __device__ constexpr int tc_na() {
  return !Fmt<F>::IQ1 || !(MODE == MODE_SEARCH || MODE == MODE_FIXED) ? 4 : (F == IQ1_M ? 8 : 6);
}
// Deferred-shift layout of the second sweep: the shifted sums are split into the entry-dependent
// part from the tensor cores, Bp' = w . h + (w/4) . g = B + Cg/4 and Bm' = B - Cg/4 (IQ1_M, whose
// shift is searched per vector), or Bd' = B + sigma Cg/4 (IQ1_S with fixed choices, whose shift
// is one per group, given or chosen by the first sweep), and a part the same for every entry of a
// vector, K(alpha, delta) = alpha Ws/64 + delta nT2, added to its best and runner-up only
// (fl(x + K) is monotone in x).  The first sweep keeps An, Cg, B.
template <int F, int MODE> __host__ __device__ constexpr bool tc_deferred(int sweep) {
  return Fmt<F>::IQ1 && (MODE == MODE_FIXED || (MODE == MODE_SEARCH && sweep == 1));
}
// Dynamic shared memory with nb buffers of the per-quad operands and state; two buffers (the
// prep warp fills quad q + 1 while the consumers sweep quad q) wherever they fit.
template <int F, int MODE> __host__ __device__ constexpr size_t tc_smem(int nb) {
  return TcCfg<F>::SMEM + (MODE == MODE_EVERY ? TcCfg<F>::EVERY : 0) +
         (size_t)nb * ((size_t)tc_na<F, MODE>() * 4096 + TcCfg<F>::STATE);
}
template <int F, int MODE> __host__ __device__ constexpr int tc_nbuf() {
  return tc_smem<F, MODE>(2) <= kMaxDynSmem ? 2 : 1;
}

template <int F, int MODE, typename TIn>
__global__ void __launch_bounds__(kTcThreads, 1) encode_tc_kernel(EncArgs a, EncWs ws, int64_t nquads) {
  constexpr int C = Fmt<F>::C, N = Fmt<F>::N, VPG = Fmt<F>::VPG, BB = Fmt<F>::BB, G = Fmt<F>::G;
  constexpr int NQ = TcCfg<F>::NQ, NCH = TcCfg<F>::NCH, NS = Fmt<F>::IQ1 ? 8 : 16;
  constexpr uint32_t IDESC = umma_idesc<kChunk>();
  extern __shared__ __align__(1024) uint8_t smem[];
  float *cb = reinterpret_cast<float *>(smem);              // codebook g [N x 8], then h [N x 8]
  float *hlo = cb + (size_t)N * 16;                         // IQ2: low tf32 part of h [N x 8]
  constexpr int NA = tc_na<F, MODE>();
  constexpr int NB = tc_nbuf<F, MODE>();
  float *aop0 = hlo + TcCfg<F>::HLO / 4;                    // [NB][NA][128 x 8] per-vector operands
  float *xchg = aop0 + NB * NA * 1024;                      // [2][128][4] float4 per-choice minima, swizzled
  // the 16-byte word w (choices 4w .. 4w + 3) of vector r in warp half h: its 128-byte segment's
  // slots permuted by (r / 4) mod 8, so that a warp reading its own rows, or the rows of its lanes'
  // groups at per-lane words, spreads over all bank groups
  auto xw = [&](int h, int r, int w) -> float4 * {
    return reinterpret_cast<float4 *>(xchg) + h * 512 + ((r * 4 + w) ^ ((r >> 2) & 7));
  };
  float4 *xchg2 = reinterpret_cast<float4 *>(xchg + 2 * 128 * 16);  // [2][128] (best, second, key)
  uint32_t *packbuf = reinterpret_cast<uint32_t *>(xchg2 + 2 * 128); // [4][24]
  float *evm = reinterpret_cast<float *>(packbuf + 4 * 24);        // [2][16][128] (every mode)
  uint32_t *evk = reinterpret_cast<uint32_t *>(evm + 2 * 128 * 16); // [2][16][128] (every mode)
  float *evt = reinterpret_cast<float *>(evk + 2 * 128 * 16);       // [2][16][128] (every mode)
  float4 *vst = reinterpret_cast<float4 *>(MODE == MODE_EVERY ? evt + 2 * 128 * 16 : evm);  // [NB][128]
  uint32_t *bst = reinterpret_cast<uint32_t *>(vst + NB * 128);     // [NB][4]
  __shared__ uint64_t cb_bar, full_bar[2], empty_bar[2], op_bar, op_full[2], op_empty[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int hsplit;  // IQ2: some h = g^2 needs its low tf32 part (read by the MMA issuer)

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool control = warp == kCtrlWarp;
  const int quarter = warp & 3, sub = warp >> 2;
  if (threadIdx.x == 0) {
    mbar_init(&full_bar[0], 1);
    mbar_init(&full_bar[1], 1);
    mbar_init(&empty_bar[0], kTcConsumers);
    mbar_init(&empty_bar[1], kTcConsumers);
    mbar_init(&op_bar, 128);  // searched IQ1_S: the 4 blocks' shifted operands (every writer), per quad
    mbar_init(&op_full[0], kPrepWarps);   // the prep warps have written a quad's operands and state
    mbar_init(&op_full[1], kPrepWarps);
    mbar_init(&op_empty[0], kTcConsumers);   // the consumers are done with a quad's buffer
    mbar_init(&op_empty[1], kTcConsumers);
    abort_flag = 0;
    mbar_fence_init();
  }
  if (control) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(TcCfg<F>::ALLOC));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const bool grid_bad = ws.hdr[0] != 0;
  const bool ok = grid_bad || load_codebook(reinterpret_cast<float4 *>(cb), ws.tab, N * 64, &cb_bar);
  if (grid_bad && blockIdx.x == 0 && threadIdx.x == 0 && a.status) atomicOr(a.status, IQ_STATUS_BAD_GRID);
  __syncthreads();
  // IQ2 codebooks: h = g^2 has up to 14 significant bits (values up to 127), tf32 holds 11.  Each
  // h becomes hi = rna_tf32(h) in place plus lo = h - hi (an integer of at most 4 significant
  // bits), both exact in tf32; when some h needs the low part, B = w . hi + w . lo takes two more
  // MMAs per chunk, so the codebook operand stays exact for every accepted grid.
  if constexpr (!Fmt<F>::IQ1) {
    bool inexact = false;
    if (ok && !grid_bad) {
      float *hs = cb + (size_t)N * 8;
      for (int i = threadIdx.x; i < N * 8; i += blockDim.x) {
        const float h = hs[i], hh = tf32_rna(h);
        inexact |= hh != h;
        hs[i] = hh;
        hlo[i] = __fsub_rn(h, hh);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    const int any = __syncthreads_or(inexact);
    if (threadIdx.x == 0) hsplit = any;
  }
  __syncthreads();  // hsplit is published

  constexpr bool kOpSync = F == IQ1_S && MODE == MODE_SEARCH;  // operands written between the sweeps
  const int g0 = lane & ~(VPG - 1);
  const int cg = lane / VPG;
  const int row = 32 * quarter + lane;                      // this lane's vector in the quad
  const uint32_t taddr = tmem + ((uint32_t)(32 * quarter) << 16);
  uint32_t cc = 0;                                          // chunk sequence number
  uint32_t issued = 0;                                      // (control) chunks committed
  uint32_t nquad = 0;                                       // (control) quads issued
  int st_acc = 0;

  bool okl = ok;                                            // this thread's waits all completed
  // A timeout in any role sets abort_flag (and the status bit); every role checks it once per quad,
  // and every wait is bounded, so all roles leave the quad loop and meet at the final barrier.
  auto give_up = [&]() {
    *(volatile int *)&abort_flag = 1;
    if (a.status && lane == 0) atomicOr(a.status, IQ_STATUS_TIMEOUT);
  };
  uint32_t it = 0;                                          // this CTA's quad counter
  if (warp >= kPrepWarp) {
    // ---- prep: loads, scale, sign rule and tf32 operands of the quad, one quad ahead; prep warp
    // pw takes blocks 2 pw and 2 pw + 1 of each quad ----------------------------------------
    const int blk0 = 2 * (warp - kPrepWarp);
    for (int64_t qd = blockIdx.x; qd < nquads; qd += gridDim.x, it++) {
      const uint32_t qb = it % NB;
      if (it >= NB && okl && !mbar_wait_bounded(&op_empty[qb], ((it / NB) - 1) & 1)) okl = false;
      okl = __all_sync(0xffffffffu, okl);
      if (!okl) { give_up(); break; }
      if (*(volatile int *)&abort_flag) break;
      float X[2][8], Wt[2][8];
      int d16p[2], chp[2];   // given scales, and (lane < G) the fixed choice of group `lane`
#pragma unroll
      for (int bi = 0; bi < 2; bi++) {   // every load first
        const int64_t b = qd * 4 + blk0 + bi;
        d16p[bi] = -1;
        chp[bi] = 0;
        if (b < a.nblocks && !grid_bad) {
          Vec t;
          load_block_vec<TIn>(a, b, lane, t);
#pragma unroll
          for (int i = 0; i < 8; i++) { X[bi][i] = t.x[i]; Wt[bi][i] = t.w[i]; }
          if (a.d16) d16p[bi] = (int)a.d16[b];
          if (MODE == MODE_FIXED && lane < G) chp[bi] = fixed_choice<G>(a, b, lane);
        }
      }
      float *aop = aop0 + qb * NA * 1024;
#pragma unroll
      for (int bi = 0; bi < 2; bi++) {
        const int blk = blk0 + bi;
        const int64_t b = qd * 4 + blk;
        const int prow = 32 * blk + lane;
        Vec v;
#pragma unroll
        for (int i = 0; i < 8; i++) { v.x[i] = X[bi][i]; v.w[i] = Wt[bi][i]; }
        int bad = 0;
        uint32_t d16 = 0;
        const bool has = b < a.nblocks && !grid_bad;
        if (has) d16 = block_scale<F, MODE>(v, lane, d16p[bi], chp[bi], bad);
        const int cfix = MODE == MODE_FIXED ? __shfl_sync(0xffffffffu, chp[bi], cg) : 0;  // this vector's group
        st_acc |= bad;
        const bool active = has && d16 != 0;
        if (active) {
          vec_setup<F>(v);
        } else if (b < a.nblocks) {
          // a rejected or zero-scale block: all-zero payload; every choice decodes to zeros
          if (MODE == MODE_EVERY) {
            for (int c = 0; c < C; c++)
              for (int i = lane; i < BB; i += 32) a.payload[((size_t)c * a.nblocks + b) * BB + i] = 0;
          } else if (MODE != MODE_TABLE) {
            for (int i = lane; i < BB; i += 32) a.payload[b * BB + i] = 0;
            if (a.wb) write_back_zero<F, TIn>(a, b, lane);
          }
          if (a.table && MODE != MODE_FIXED) {
            float cs = 0.0f;
            if (has) {
#pragma unroll
              for (int i = 0; i < 8; i++) cs = __fmaf_rn(__fmul_rn(v.w[i], v.x[i]), v.x[i], cs);
            }
            const float e0 = group_sum<VPG>(cs, g0);
            const float val = (bad || grid_bad) ? __int_as_float(0x7fc00000) : e0;
            if (lane == g0)
              for (int c = 0; c < C; c++) a.table[(b * G + cg) * C + c] = val;
          }
        }
        // IQ1_S with fixed choices: the sign of the group's shift (choice c = scale + 8 * shift bit)
        const float sig = MODE == MODE_FIXED && NA == 6 && active && (cfix >> 3) ? -0.25f : 0.25f;
#pragma unroll
        for (int k = 0; k < 8; k++) {
          const float nw = active ? v.nw2[k] : 0.0f, ww = active ? v.w[k] : 0.0f;
          const float nh = tf32_rna(nw), wh = tf32_rna(ww);
          aop[0 * 1024 + kmaj(prow, k)] = nh;
          aop[1 * 1024 + kmaj(prow, k)] = tf32_rna(__fsub_rn(nw, nh));
          const float wl = tf32_rna(__fsub_rn(ww, wh));
          aop[2 * 1024 + kmaj(prow, k)] = wh;
          aop[3 * 1024 + kmaj(prow, k)] = wl;
          if (NA == 8) {  // exact power-of-two scalings of the tf32 parts
            aop[4 * 1024 + kmaj(prow, k)] = 0.25f * wh;
            aop[5 * 1024 + kmaj(prow, k)] = 0.25f * wl;
            aop[6 * 1024 + kmaj(prow, k)] = -0.25f * wh;
            aop[7 * 1024 + kmaj(prow, k)] = -0.25f * wl;
          } else if (NA == 6 && MODE == MODE_FIXED) {
            aop[4 * 1024 + kmaj(prow, k)] = sig * wh;
            aop[5 * 1024 + kmaj(prow, k)] = sig * wl;
          }
        }
        // .w: the sign mask (bits 0..7) and, with fixed choices, the group's choice (bits 8..15)
        vst[qb * 128 + prow] = active ? make_float4(v.Cs, v.nT2, v.Ws, __int_as_float(v.sgn | cfix << 8))
                                      : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (lane == 0) bst[qb * 4 + blk] = d16 | (active ? 1u << 16 : 0u);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // operands seen by the MMAs
      __syncwarp();
      if (lane == 0) mbar_arrive(&op_full[qb]);
    }
  } else if (control) {
    // IQ2: whether B takes the low parts of h too (read once: the flag is fixed for the call)
    const bool hsreg = !Fmt<F>::IQ1 && *(volatile int *)&hsplit;
    // ---- MMA issue: sweep 1 (unless fixed choices) and sweep 2 (unless table only) ---------
    for (int64_t qd = blockIdx.x; qd < nquads; qd += gridDim.x, it++) {
      const uint32_t qb = it % NB;
      if (lane == 0) {
        if (okl && !mbar_wait_bounded(&op_full[qb], (it / NB) & 1)) okl = false;
        if (okl && !*(volatile int *)&abort_flag) {
            const int nsweeps = (MODE != MODE_FIXED) + (MODE != MODE_TABLE);
            const uint32_t sa = smem_u32(aop0 + qb * NA * 1024), sg = smem_u32(cb), sh = sg + N * 32, shl = smem_u32(hlo);
            for (int sw = 0; sw < nsweeps; sw++) {
              for (int ch = 0; ch < NCH; ch++, issued++) {
                const uint32_t buf = issued & 1;
                // searched IQ1_S: the second sweep's shifted operands are written after the first sweep
                if (kOpSync && sw == 1 && ch == 0 && okl && !mbar_wait_bounded(&op_bar, nquad & 1)) okl = false;
                if (!okl || (issued >= 2 && !mbar_wait_bounded(&empty_bar[buf], ((issued >> 1) - 1) & 1))) {
                  okl = false;  // stop issuing; consumers' waits on the missing chunks time out
                  break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * NQ * kChunk;
                const uint64_t bg = umma_desc(sg + ch * kChunk * 32), bh = umma_desc(sh + ch * kChunk * 32);
                umma_tf32(d, umma_desc(sa + 0 * 4096), bg, IDESC, 0);          // An = nw2 . g
                umma_tf32(d, umma_desc(sa + 1 * 4096), bg, IDESC, 1);
                if (tc_deferred<F, MODE>(sw) && F == IQ1_S) {
                  umma_tf32(d + kChunk, umma_desc(sa + 2 * 4096), bh, IDESC, 0);      // Bd' = w . h
                  umma_tf32(d + kChunk, umma_desc(sa + 3 * 4096), bh, IDESC, 1);
                  umma_tf32(d + kChunk, umma_desc(sa + 4 * 4096), bg, IDESC, 1);      //      + (sigma w/4) . g
                  umma_tf32(d + kChunk, umma_desc(sa + 5 * 4096), bg, IDESC, 1);
                } else if (tc_deferred<F, MODE>(sw)) {
                  umma_tf32(d + kChunk, umma_desc(sa + 2 * 4096), bh, IDESC, 0);      // Bp' = w . h
                  umma_tf32(d + kChunk, umma_desc(sa + 3 * 4096), bh, IDESC, 1);
                  umma_tf32(d + kChunk, umma_desc(sa + 4 * 4096), bg, IDESC, 1);      //      + (w/4) . g
                  umma_tf32(d + kChunk, umma_desc(sa + 5 * 4096), bg, IDESC, 1);
                  umma_tf32(d + 2 * kChunk, umma_desc(sa + 2 * 4096), bh, IDESC, 0);  // Bm' = w . h
                  umma_tf32(d + 2 * kChunk, umma_desc(sa + 3 * 4096), bh, IDESC, 1);
                  umma_tf32(d + 2 * kChunk, umma_desc(sa + 6 * 4096), bg, IDESC, 1);  //      - (w/4) . g
                  umma_tf32(d + 2 * kChunk, umma_desc(sa + 7 * 4096), bg, IDESC, 1);
                } else {
                  if (NQ == 3) {
                    umma_tf32(d + kChunk, umma_desc(sa + 2 * 4096), bg, IDESC, 0);  // Cg = w . g
                    umma_tf32(d + kChunk, umma_desc(sa + 3 * 4096), bg, IDESC, 1);
                  }
                  umma_tf32(d + (NQ - 1) * kChunk, umma_desc(sa + 2 * 4096), bh, IDESC, 0);  // B = w . h
                  umma_tf32(d + (NQ - 1) * kChunk, umma_desc(sa + 3 * 4096), bh, IDESC, 1);
                  if (hsreg) {                                                              //   + w . h lo
                    const uint64_t bl = umma_desc(shl + ch * kChunk * 32);
                    umma_tf32(d + (NQ - 1) * kChunk, umma_desc(sa + 2 * 4096), bl, IDESC, 1);
                    umma_tf32(d + (NQ - 1) * kChunk, umma_desc(sa + 3 * 4096), bl, IDESC, 1);
                  }
                }
                umma_commit(&full_bar[buf]);
              }
              if (!okl) break;
            }
        }
        nquad++;
      }
      okl = __shfl_sync(0xffffffffu, okl, 0);
      if (!okl) { give_up(); break; }
      if (*(volatile int *)&abort_flag) break;
    }
  } else {
  for (int64_t qd = blockIdx.x; qd < nquads; qd += gridDim.x, it++) {
    const uint32_t qb = it % NB;
    if (okl && !mbar_wait_bounded(&op_full[qb], (it / NB) & 1)) okl = false;
    okl = __all_sync(0xffffffffu, okl);
    if (!okl) { give_up(); break; }
    if (*(volatile int *)&abort_flag) break;
    const int64_t b = qd * 4 + quarter;
    const uint32_t bs = bst[qb * 4 + quarter];
    const uint32_t d16 = bs & 0xffffu;
    const bool active = (bs >> 16) & 1u;
    const float4 vs = vst[qb * 128 + row];
    const float vCs = vs.x, vnT2 = vs.y, vWs = vs.z;
    const int vsgn = __float_as_int(vs.w) & 0xff;
    const int vfix = __float_as_int(vs.w) >> 8;   // fixed-choice mode: the group's choice
    const float Cgrp = group_sum<VPG>(vCs, g0);
    float *aop = aop0 + qb * NA * 1024;

    // ---- consumers ---------------------------------------------------------------------------
    const float d = half_bits_to_float((uint16_t)d16);
    const IQ1Const kc = iq1_consts();
    const uint64_t nT2p = pk2(vnT2, vnT2), Wsp = pk2(vWs, vWs);
    const float w64 = 0.015625f * vWs, t8 = 0.125f * vnT2;  // exact power-of-two scalings
    const int ebase0 = 32 * sub;  // this warp's first entry in each chunk
    // IQ1_S second sweep (fixed or searched choices): deferred layout [An | Bd' | -]
    constexpr bool kDefS = F == IQ1_S && (MODE == MODE_FIXED || MODE == MODE_SEARCH);
    // waits for chunk `cc`, hands the warp's 2 x 16 columns to fn(half, An, Cg, B), releases it
    // (after a timeout the remaining chunks are skipped without waiting); two_cols: the chunk has
    // only the first two columns (the IQ1_S deferred second sweep)
    auto run_chunk = [&](auto two_cols, auto &&fn) {
      const uint32_t buf = cc & 1;
      if (okl && !mbar_wait_bounded(&full_bar[buf], (cc >> 1) & 1)) okl = false;
      okl = __all_sync(0xffffffffu, okl);
      tc_fence_after();
      const uint32_t col = buf * NQ * kChunk + ebase0;
#pragma unroll
      for (int h = 0; h < 2; h++) {
        float An[16], Bq[16], Cq[16];
        tmem_ld16(taddr + col + 16 * h, An);
        if (NQ == 3) tmem_ld16(taddr + col + kChunk + 16 * h, Cq);
        if constexpr (!decltype(two_cols)::value) tmem_ld16(taddr + col + (NQ - 1) * kChunk + 16 * h, Bq);
        tmem_wait_ld();
        if (active && okl) fn(h, An, Cq, Bq);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[buf]);
      cc++;
    };

    int c1 = 0;
    bool gflag = false;
    float smin = 0.0f;  // searched mode: this vector's minimum score under c1 (from sweep 1)
    uint64_t alp[NS];
#pragma unroll
    for (int s = 0; s < NS; s++) { const float al = alpha_of<F>(d, s); alp[s] = pk2(al, al); }
    if (MODE != MODE_FIXED) {
      float m[C];
#pragma unroll
      for (int c = 0; c < C; c++) m[c] = INFINITY;
      for (int ch = 0; ch < NCH; ch++) {
        run_chunk(std::false_type{}, [&](int h, const float *An, const float *Cq, const float *Bq) {
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const uint64_t A2 = pk2(An[2 * i], An[2 * i + 1]), B2 = pk2(Bq[2 * i], Bq[2 * i + 1]);
            if (!Fmt<F>::IQ1) {
#pragma unroll
              for (int c = 0; c < C; c++) {
                const float2 sc = up2(ffma2(alp[c], B2, A2));
                m[c] = min3f(m[c], sc.x, sc.y);
              }
            } else {
              const uint64_t C2 = pk2(Cq[2 * i], Cq[2 * i + 1]);
              const uint64_t Anp = ffma2(kc.p125, nT2p, A2), Anm = ffma2(kc.m125, nT2p, A2);
              const uint64_t Bw = ffma2(kc.w64, Wsp, B2);
              const uint64_t Bp = ffma2(kc.p025, C2, Bw), Bm = ffma2(kc.m025, C2, Bw);
#pragma unroll
              for (int s = 0; s < 8; s++) {
                const float2 sp = up2(ffma2(alp[s], Bp, Anp)), sm = up2(ffma2(alp[s], Bm, Anm));
                if (F == IQ1_S) {
                  m[s] = min3f(m[s], sp.x, sp.y);
                  m[8 + s] = min3f(m[8 + s], sm.x, sm.y);
                } else {
                  m[s] = min3f(min3f(m[s], sp.x, sp.y), sm.x, sm.y);
                }
              }
            }
          }
        });
      }
      // minima of the two consumer warps of this block
      // 4 choices per 16-byte word, lanes on consecutive words: one conflict-free vector store each
#pragma unroll
      for (int c = 0; c < C; c += 4) *xw(sub, row, c / 4) = make_float4(m[c], m[c + 1], m[c + 2], m[c + 3]);
      named_bar(2, kTcConsumers * 32);
      if constexpr (MODE == MODE_EVERY) {
#pragma unroll
        for (int c = 0; c < C; c += 4) {
          const float4 u = *xw(0, row, c / 4), v = *xw(1, row, c / 4);
          m[c] = fminf(u.x, v.x); m[c + 1] = fminf(u.y, v.y); m[c + 2] = fminf(u.z, v.z); m[c + 3] = fminf(u.w, v.w);
        }
        // every choice's minimum and the bound above it that holds every candidate whose error
        // could be within the near-tie margin of the minimum (as in the searched second sweep)
#pragma unroll
        for (int c = 0; c < C; c++) {
          const float al = alpha_choice<F>(d, c);
          const float e1 = __fmul_rn(al, m[c]);
          const float De = 1.01f * kMargin * fmaxf(4.0f * vCs + 2.0f * e1, 0.0f);
          evt[(sub * 16 + c) * 128 + row] =
              active ? m[c] + 1.01f * (De / al) + 9.5367431640625e-07f * fabsf(m[c]) : -INFINITY;
          evm[(sub * 16 + c) * 128 + row] = m[c];
          evk[(sub * 16 + c) * 128 + row] = 0xffffu;  // no key yet, no near candidate
        }
      } else if (active) {
        // the group's VPG lanes share its choices: lane kq forms the group errors of choices
        // kq * CPL .. kq * CPL + CPL - 1 (the group's minima of both warps, summed in vector order),
        // then the lanes merge (least error, lowest choice on equal errors, and the runner-up)
        constexpr int CPL = C / VPG;
        static_assert(CPL % 4 == 0, "whole 16-byte words of choices");
        const int kq = lane - g0;
        float D1 = INFINITY, D2 = INFINITY;
#pragma unroll
        for (int j = 0; j < CPL; j += 4) {
          const int cw = (kq * CPL + j) / 4;   // the 16-byte word of these 4 choices
          float4 S;
#pragma unroll
          for (int v = 0; v < VPG; v++) {
            const int rv = 32 * quarter + g0 + v;
            const float4 u = *xw(0, rv, cw), w = *xw(1, rv, cw);
            const float4 mv = make_float4(fminf(u.x, w.x), fminf(u.y, w.y), fminf(u.z, w.z), fminf(u.w, w.w));
            S = v == 0 ? mv : make_float4(__fadd_rn(S.x, mv.x), __fadd_rn(S.y, mv.y), __fadd_rn(S.z, mv.z), __fadd_rn(S.w, mv.w));
          }
          const float Sv[4] = {S.x, S.y, S.z, S.w};
#pragma unroll
          for (int t = 0; t < 4; t++) {
            const int c = kq * CPL + j + t;
            const float D = __fmul_rn(alpha_of<F>(d, F == IQ1_S ? (c & 7) : c), Sv[t]);
            if (a.table && sub == 0) a.table[(b * G + cg) * C + c] = __fadd_rn(Cgrp, D);
            D2 = fminf(D2, fmaxf(D1, D));
            if (D < D1) { D1 = D; c1 = c; }
          }
        }
#pragma unroll
        for (int off = 1; off < VPG; off <<= 1) {
          const float oD1 = __shfl_xor_sync(0xffffffffu, D1, off), oD2 = __shfl_xor_sync(0xffffffffu, D2, off);
          const int oc = __shfl_xor_sync(0xffffffffu, c1, off);
          D2 = fminf(fmaxf(D1, oD1), fminf(D2, oD2));
          if (oD1 < D1 || (oD1 == D1 && oc < c1)) { D1 = oD1; c1 = oc; }
        }
        smin = fminf(reinterpret_cast<const float *>(xw(0, row, c1 / 4))[c1 & 3],
                     reinterpret_cast<const float *>(xw(1, row, c1 / 4))[c1 & 3]);
        gflag = __fsub_rn(D2, D1) <= kMargin * (4.0f * Cgrp + D1 + D2);
      }
    } else if (active) {
      c1 = vfix;
    }
    if constexpr (kOpSync) {
      // the second sweep's shifted operand sigma w/4 (hi, lo) of each vector, sigma the sign of its
      // group's chosen shift; the control warp issues the second sweep once all 4 blocks are in
      if (sub == 0) {
        const float sig = (c1 >> 3) ? -0.25f : 0.25f;
#pragma unroll
        for (int k = 0; k < 8; k++) {   // the tf32 parts of w (zero for an inactive block), scaled
          aop[4 * 1024 + kmaj(row, k)] = sig * aop[2 * 1024 + kmaj(row, k)];
          aop[5 * 1024 + kmaj(row, k)] = sig * aop[3 * 1024 + kmaj(row, k)];
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&op_bar);
      }
    }

    if constexpr (MODE == MODE_EVERY) {
      // ---- sweep 2 (every choice): each vector's best candidate under every choice ---------
      // A part of the sweep (16 entries of the warp) goes through the exact bookkeeping for a
      // choice only when the part's minimum under that choice is at most T[c]: the key of the
      // minimum (the lowest entry whose score equals it exactly; the same MMAs and rounded packed
      // FMAs reproduce sweep 1's values) and the number of candidates at most T[c] (two or more
      // mean a near tie, which the exact rescoring re-decides under that choice).
      // this vector's entries, choice c at [128 c] (lanes on consecutive banks)
      const float *mrow = evm + sub * 16 * 128 + row;
      const float *trow = evt + sub * 16 * 128 + row;
      uint32_t *krow = evk + sub * 16 * 128 + row;
      for (int ch = 0; ch < NCH; ch++) {
        const int eb = ch * kChunk + ebase0;
        run_chunk(std::false_type{}, [&](int h, const float *An, const float *Cq, const float *Bq) {
          float mn[C];
#pragma unroll
          for (int c = 0; c < C; c++) mn[c] = INFINITY;
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const uint64_t A2 = pk2(An[2 * i], An[2 * i + 1]), B2 = pk2(Bq[2 * i], Bq[2 * i + 1]);
            if (!Fmt<F>::IQ1) {
#pragma unroll
              for (int c = 0; c < C; c++) {
                const float2 sc = up2(ffma2(alp[c], B2, A2));
                mn[c] = min3f(mn[c], sc.x, sc.y);
              }
            } else {
              const uint64_t C2 = pk2(Cq[2 * i], Cq[2 * i + 1]);
              const uint64_t Anp = ffma2(kc.p125, nT2p, A2), Anm = ffma2(kc.m125, nT2p, A2);
              const uint64_t Bw = ffma2(kc.w64, Wsp, B2);
              const uint64_t Bp = ffma2(kc.p025, C2, Bw), Bm = ffma2(kc.m025, C2, Bw);
#pragma unroll
              for (int s = 0; s < 8; s++) {
                const float2 sp = up2(ffma2(alp[s], Bp, Anp)), sm = up2(ffma2(alp[s], Bm, Anm));
                if (F == IQ1_S) {
                  mn[s] = min3f(mn[s], sp.x, sp.y);
                  mn[8 + s] = min3f(mn[8 + s], sm.x, sm.y);
                } else {
                  mn[s] = min3f(min3f(mn[s], sp.x, sp.y), sm.x, sm.y);
                }
              }
            }
          }
          uint32_t hits = 0;  // choices whose minimum over this part is within the near bound
#pragma unroll
          for (int c = 0; c < C; c += 4) {
            const float4 t4 = make_float4(trow[128 * c], trow[128 * (c + 1)], trow[128 * (c + 2)], trow[128 * (c + 3)]);
            hits |= (mn[c] <= t4.x ? 1u : 0u) << c | (mn[c + 1] <= t4.y ? 2u : 0u) << c |
                    (mn[c + 2] <= t4.z ? 4u : 0u) << c | (mn[c + 3] <= t4.w ? 8u : 0u) << c;
          }
          while (hits) {
            const int c = __ffs(hits) - 1;
            hits &= hits - 1u;
            const float Tc = trow[128 * c], mc = mrow[128 * c];
            uint32_t key = krow[128 * c] & 0xffffu, cnt = krow[128 * c] >> 16;
            const int sc = F == IQ1_S ? (c & 7) : c;
            const int db = F == IQ1_S ? (c >> 3) : 0;
            const float alf = alpha_of<F>(d, sc);  // as alp[sc]
            const uint64_t al2 = pk2(alf, alf);
#pragma unroll
            for (int i = 0; i < 8; i++) {
              const int e0 = eb + 16 * h + 2 * i;
              const uint64_t A2 = pk2(An[2 * i], An[2 * i + 1]), B2 = pk2(Bq[2 * i], Bq[2 * i + 1]);
              float2 q0, q1 = make_float2(INFINITY, INFINITY);
              if (!Fmt<F>::IQ1) {
                q0 = up2(ffma2(al2, B2, A2));
              } else {
                const uint64_t C2 = pk2(Cq[2 * i], Cq[2 * i + 1]);
                const uint64_t Bw = ffma2(kc.w64, Wsp, B2);
                if (F == IQ1_S) {
                  const uint64_t Ad = ffma2(db ? kc.m125 : kc.p125, nT2p, A2);
                  const uint64_t Bd = ffma2(db ? kc.m025 : kc.p025, C2, Bw);
                  q0 = up2(ffma2(al2, Bd, Ad));
                } else {
                  const uint64_t Anp = ffma2(kc.p125, nT2p, A2), Anm = ffma2(kc.m125, nT2p, A2);
                  const uint64_t Bp = ffma2(kc.p025, C2, Bw), Bm = ffma2(kc.m025, C2, Bw);
                  q0 = up2(ffma2(al2, Bp, Anp));
                  q1 = up2(ffma2(al2, Bm, Anm));
                }
              }
              const float vv[4] = {q0.x, q0.y, q1.x, q1.y};
              const uint32_t kk[4] = {(uint32_t)e0, (uint32_t)e0 + 1u, (uint32_t)(N + e0), (uint32_t)(N + e0) + 1u};
#pragma unroll
              for (int t = 0; t < (F == IQ1_M ? 4 : 2); t++) {
                if (vv[t] <= Tc) {
                  cnt++;
                  if (vv[t] == mc && kk[t] < key) key = kk[t];
                }
              }
            }
            krow[128 * c] = key | (min(cnt, 3u) << 16);
          }
        });
      }
      named_bar(2, kTcConsumers * 32);  // both warps' keys and counts are in shared memory
      if (sub == 0 && active) {
        uint32_t *pb = packbuf + quarter * 24;
        for (int c = 0; c < C; c++) {
          const uint32_t w0 = evk[c * 128 + row], w1 = evk[(16 + c) * 128 + row];
          const uint32_t key = min(w0 & 0xffffu, w1 & 0xffffu);
          const uint32_t cnt = (w0 >> 16) + (w1 >> 16);
          // near ties under choice c: one item (block | c << 27, vectors) for the exact rescoring
          const uint32_t vflags = __ballot_sync(0xffffffffu, cnt >= 2 || key == 0xffffu);
          if (vflags && lane == 0) {
            const int slot = atomicAdd(&ws.hdr[1], 1);
            ws.fb[slot] = make_uint2((uint32_t)b | ((uint32_t)c << 27), vflags);
          }
          if (lane < 24) pb[lane] = 0u;
          __syncwarp();
          const int k = key == 0xffffu ? 0 : (int)key;
          const int idx = F == IQ1_M ? (k % N) : k;
          const Bits lo = f_idx_lo<F>(lane);
          put_bits(pb, lo, (uint32_t)idx);
          if (F == IQ2_S || Fmt<F>::IQ1) put_bits(pb, f_idx_hi<F>(lane), (uint32_t)idx >> lo.width);
          if (!Fmt<F>::IQ1) put_bits(pb, f_sign<F>(lane), (uint32_t)vsgn);
          if (F == IQ1_M) {
            put_bits(pb, f_dbit_vec<F>(lane), (uint32_t)(k / N));
            if (lane < 4) put_bits(pb, f_d16_nib<F>(lane), (d16 >> (4 * lane)) & 15u);
          } else if (lane == 0) {
            put_bits(pb, f_d16<F>(), d16);
          }
          if (lane == g0) {
            put_bits(pb, f_scale<F>(cg), (uint32_t)(F == IQ1_S ? (c & 7) : c));
            if (F == IQ1_S) put_bits(pb, f_dbit_grp<F>(cg), (uint32_t)(c >> 3));
          }
          __syncwarp();
          const uint8_t *pbytes = reinterpret_cast<const uint8_t *>(pb);
          uint8_t *dst = a.payload + ((size_t)c * a.nblocks + b) * BB;
          for (int i = lane; i < BB; i += 32) dst[i] = pbytes[i];
          __syncwarp();
        }
      }
    } else if (MODE != MODE_TABLE) {
      // ---- sweep 2: best candidate and runner-up under choice c1 ---------------------------
      // Fixed choices: every candidate goes through the best / runner-up tracking.  Searched
      // mode: sweep 1 already gave the minimum s1 (the same MMAs and the same rounded packed
      // FMAs reproduce it exactly), so a part of the sweep is tracked only when one of its
      // scores is at most T, a bound just above s1.  Every candidate that could flag the vector (gap of the
      // errors alpha * s within the margin) lies below T; the rest cannot be the best and
      // cannot flag, so skipping them leaves the key and the flag unchanged.
      const float alpha = alpha_choice<F>(d, c1);
      const uint64_t al = pk2(alpha, alpha);
      const int dbit = F == IQ1_S ? (c1 >> 3) : 0;
      const uint64_t dA = dbit ? kc.m125 : kc.p125, dB = dbit ? kc.m025 : kc.p025;
      // Deferred layouts (IQ1_M; IQ1_S with fixed choices): raw scores alpha Bd' + An per shift;
      // the shift's K is added to the tracked best and runner-up at the end
      float Kp = 0.0f, Km = 0.0f;
      if (F == IQ1_M && active) { Kp = __fmaf_rn(alpha, w64, t8); Km = __fmaf_rn(alpha, w64, -t8); }
      if (kDefS && active) Kp = __fmaf_rn(alpha, w64, dbit ? -t8 : t8);
      // (With 256 or 512 entries nearly every part holds some lane's best, so the small codebooks
      // track everything.)
      constexpr bool kFind = MODE == MODE_SEARCH && N >= 1024;
      float T = INFINITY;
      if (kFind && active) {
        // flag iff e2 - e1 <= kMargin (4 Cs + e1 + e2), i.e. e2 - e1 <= kMargin (4 Cs + 2 e1) /
        // (1 - kMargin); the factors 1.01 and the relative term cover fp32 rounding here.  The IQ1
        // second sweeps evaluate the shifted scores in another order of rounding than the first
        // (each within the rounding bound of the margin), so their bound is twice as wide.
        constexpr float kW = Fmt<F>::IQ1 ? 2.02f : 1.01f;
        constexpr float kR = Fmt<F>::IQ1 ? 1.9073486328125e-06f : 9.5367431640625e-07f;
        const float e1 = __fmul_rn(alpha, smin);
        const float De = 1.01f * kMargin * fmaxf(4.0f * vCs + 2.0f * e1, 0.0f);
        T = smin + kW * (De / alpha) + kR * fabsf(smin);
      }
      // Two trackers per shift, over the even and the odd pairs of each half chunk (two shorter
      // dependency chains), merged below: the lower score, on equal scores the lower key (each
      // tracker keeps the first of its equal scores, and its keys only grow).
      float best = INFINITY, second = INFINITY, bestm = INFINITY, secondm = INFINITY;
      float best1 = INFINITY, second1 = INFINITY, bestm1 = INFINITY, secondm1 = INFINITY;
      int key = 0, keym = 0, key1 = 0, keym1 = 0;
      constexpr int PPH = F == IQ1_M ? 16 : 8;  // candidate pairs per half chunk
      for (int ch = 0; ch < NCH; ch++) {
        const int eb = ch * kChunk + ebase0;
        run_chunk(std::integral_constant<bool, kDefS>{}, [&](int h, const float *An, const float *Cq, const float *Bq) {
          uint64_t sc[PPH];  // pair p: entries e0, e0 + 1 (IQ1_M: p >= 8 the minus shift)
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const uint64_t A2 = pk2(An[2 * i], An[2 * i + 1]);
            if (kDefS) {
              sc[i] = ffma2(al, pk2(Cq[2 * i], Cq[2 * i + 1]), A2);
              continue;
            }
            const uint64_t B2 = pk2(Bq[2 * i], Bq[2 * i + 1]);
            if (!Fmt<F>::IQ1) {
              sc[i] = ffma2(al, B2, A2);
            } else if (F == IQ1_S) {
              const uint64_t C2 = pk2(Cq[2 * i], Cq[2 * i + 1]);
              const uint64_t Bw = ffma2(kc.w64, Wsp, B2);
              const uint64_t Ad = ffma2(dA, nT2p, A2), Bd = ffma2(dB, C2, Bw);
              sc[i] = ffma2(al, Bd, Ad);
            } else {
              // deferred layout: the second column holds Bp', the third Bm'
              const uint64_t P2 = pk2(Cq[2 * i], Cq[2 * i + 1]);
              sc[i] = ffma2(al, P2, A2);
              sc[8 + i] = ffma2(al, B2, A2);
            }
          }
          if (kFind) {
            float mn = INFINITY, mnm = INFINITY;
#pragma unroll
            for (int p = 0; p < 8; p++) {
              const float2 q = up2(sc[p]);
              mn = min3f(mn, q.x, q.y);
              if (F == IQ1_M) { const float2 r = up2(sc[8 + p]); mnm = min3f(mnm, r.x, r.y); }
            }
            const bool hit = F == IQ1_M ? (__fadd_rn(mn, Kp) <= T || __fadd_rn(mnm, Km) <= T)
                                        : (kDefS ? __fadd_rn(mn, Kp) <= T : mn <= T);
            if (!hit) return;
          }
#pragma unroll
          for (int p = 0; p < 8; p += 2) {
            const int e0 = eb + 16 * h + 2 * p;
            track2(up2(sc[p]), e0, best, second, key);
            track2(up2(sc[p + 1]), e0 + 2, best1, second1, key1);
            if (F == IQ1_M) {
              track2(up2(sc[8 + p]), N + e0, bestm, secondm, keym);
              track2(up2(sc[9 + p]), N + e0 + 2, bestm1, secondm1, keym1);
            }
          }
        });
      }
      merge_track(best, second, key, best1, second1, key1);
      if (F == IQ1_M) merge_track(bestm, secondm, keym, bestm1, secondm1, keym1);
      if (kDefS) {  // back to full scores (INFINITY stays INFINITY)
        best = __fadd_rn(best, Kp);
        second = __fadd_rn(second, Kp);
      }
      if (F == IQ1_M) {  // back to full scores (INFINITY stays INFINITY)
        best = __fadd_rn(best, Kp);
        second = __fadd_rn(second, Kp);
        const float bm = __fadd_rn(bestm, Km), sm2 = __fadd_rn(secondm, Km);
        const bool takem = bm < best;  // equal scores keep the plus shift (its keys are lower)
        second = min3f(second, sm2, takem ? best : bm);
        if (takem) { best = bm; key = keym; }
      }
      xchg2[sub * 128 + row] = make_float4(best, second, __int_as_float(key), 0.0f);
      named_bar(2, kTcConsumers * 32);
      if (sub == 0 && active) {
        const float4 o0 = xchg2[row], o1 = xchg2[128 + row];
        const int k0 = __float_as_int(o0.z), k1 = __float_as_int(o1.z);
        const bool first = o0.x < o1.x || (o0.x == o1.x && k0 < k1);
        const float s1 = fminf(o0.x, o1.x);
        const float s2 = min3f(fmaxf(o0.x, o1.x), o0.y, o1.y);
        key = first ? k0 : k1;
        const float e1 = __fmul_rn(alpha, s1), e2 = __fmul_rn(alpha, s2);
        // searched mode: no second candidate near the best means no flag; no best found at all
        // (cannot happen while both sweeps agree) hands the vector to the exact rescoring
        const bool vflag = !(s1 < INFINITY) ||
                           (s2 < INFINITY && __fsub_rn(e2, e1) <= kMargin * (4.0f * vCs + e1 + e2));
        // pack
        uint32_t *pb = packbuf + quarter * 24;
        if (lane < 24) pb[lane] = 0u;
        __syncwarp();
        const int idx = F == IQ1_M ? (key % N) : key;
        const Bits lo = f_idx_lo<F>(lane);
        put_bits(pb, lo, (uint32_t)idx);
        if (F == IQ2_S || Fmt<F>::IQ1) put_bits(pb, f_idx_hi<F>(lane), (uint32_t)idx >> lo.width);
        if (!Fmt<F>::IQ1) put_bits(pb, f_sign<F>(lane), (uint32_t)vsgn);
        if (F == IQ1_M) {
          put_bits(pb, f_dbit_vec<F>(lane), (uint32_t)(key / N));
          if (lane < 4) put_bits(pb, f_d16_nib<F>(lane), (d16 >> (4 * lane)) & 15u);
        } else if (lane == 0) {
          put_bits(pb, f_d16<F>(), d16);
        }
        if (lane == g0) {
          put_bits(pb, f_scale<F>(cg), (uint32_t)(F == IQ1_S ? (c1 & 7) : c1));
          if (F == IQ1_S) put_bits(pb, f_dbit_grp<F>(cg), (uint32_t)(c1 >> 3));
        }
        __syncwarp();
        const uint8_t *pbytes = reinterpret_cast<const uint8_t *>(pb);
        for (int i = lane; i < BB; i += 32) a.payload[b * BB + i] = pbytes[i];
        __syncwarp();
        const uint32_t flags = __ballot_sync(0xffffffffu, gflag || vflag);
        if (flags && lane == 0) {
          const int slot = atomicAdd(&ws.hdr[1], 1);
          ws.fb[slot] = make_uint2((uint32_t)b, flags);
        }
        // write-back: a block left to the exact rescoring is written by it, after its final
        // decisions (it reads the block's weight first)
        if (a.wb && !flags) {
          float g8[8];
#pragma unroll
          for (int i = 0; i < 8; i++) g8[i] = cb[kmaj(idx, i)];
          write_back_vec<F, TIn>(a, b, lane, g8, d, F == IQ1_S ? (c1 & 7) : c1, vsgn,
                                 F == IQ1_S ? (c1 >> 3) : F == IQ1_M ? key / N : 0);
        }
      }
    }
    // this warp is done with the quad's state and operands (its MMAs have completed): the prep
    // warp may refill the buffer
    __syncwarp();
    if (lane == 0) mbar_arrive(&op_empty[qb]);
  }
  }
  if (!okl && a.status) atomicOr(a.status, IQ_STATUS_TIMEOUT);
  if (st_acc && a.status && lane == 0) atomicOr(a.status, st_acc);
  // every committed chunk must have completed before tensor memory is released
  if (control && lane == 0) {
    for (uint32_t u = issued >= 2 ? issued - 2 : 0; u < issued; u++) mbar_wait_bounded(&full_bar[u & 1], (u >> 1) & 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (control) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TcCfg<F>::ALLOC));
}

// ---------------------------------------------------------------------------------------------
// Exact rescoring of flagged groups.
template <int F>
__device__ __forceinline__ double exact_err(const float *x, const float *w, const Entry &en, float d, int s, int sgn,
                                            int dbit) {
  double acc = 0.0;
  if (!Fmt<F>::IQ1) {
    const float dl = __fmul_rn(__fmul_rn(d, (float)(2 * s + 1)), 0.125f);
#pragma unroll
    for (int i = 0; i < 8; i++) {
      float q = __fmul_rn(dl, en.g[i]);
      q = ((sgn >> i) & 1) ? -q : q;
      const double df = __dsub_rn((double)x[i], (double)q);
      acc = __dadd_rn(acc, __dmul_rn((double)w[i], __dmul_rn(df, df)));
    }
  } else {
    const float dl = __fmul_rn(d, (float)(2 * s + 1));
    const float delta = dbit ? -0.125f : 0.125f;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const float q = __fmul_rn(dl, __fadd_rn(en.g[i], delta));
      const double df = __dsub_rn((double)x[i], (double)q);
      acc = __dadd_rn(acc, __dmul_rn((double)w[i], __dmul_rn(df, df)));
    }
  }
  return acc;
}

__device__ __forceinline__ Vec shfl_vec(const Vec &v, int src) {
  Vec r;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    r.x[i] = __shfl_sync(0xffffffffu, v.x[i], src);
    r.w[i] = __shfl_sync(0xffffffffu, v.w[i], src);
    r.nw2[i] = __shfl_sync(0xffffffffu, v.nw2[i], src);
  }
  r.Cs = __shfl_sync(0xffffffffu, v.Cs, src);
  r.nT2 = __shfl_sync(0xffffffffu, v.nT2, src);
  r.Ws = __shfl_sync(0xffffffffu, v.Ws, src);
  r.sgn = __shfl_sync(0xffffffffu, v.sgn, src);
  return r;
}

// the fp32 score of candidate (entry en, delta bit db) under alpha, computed exactly as the sweep does
template <int F>
__device__ __forceinline__ float cand_score(const Vec &v, const Entry &en, float alpha, int db) {
  if (!Fmt<F>::IQ1) {
    float An, B;
    ab2(v.nw2, v.w, en, An, B);
    return __fmaf_rn(alpha, B, An);
  } else {
    float Anp, Bp, Anm, Bm;
    ab1(v, en, Anp, Bp, Anm, Bm);
    return db ? __fmaf_rn(alpha, Bm, Anm) : __fmaf_rn(alpha, Bp, Anp);
  }
}

template <int F>
__device__ __forceinline__ void cand_of_choice(int c, int &s, int &db0, int &db1) {
  if (F == IQ1_S) { s = c & 7; db0 = db1 = c >> 3; }
  else if (F == IQ1_M) { s = c; db0 = 0; db1 = 1; }
  else { s = c; db0 = db1 = 0; }
}

// Write-back of a rescored block from its final payload bytes (one warp; lane = vector), with the
// codebook values from the prepared table.
template <int F, typename TIn>
__device__ __forceinline__ void write_back_bytes(const EncArgs &a, const float4 *tab, int64_t b, int lane,
                                                 const uint8_t *pbytes, float d) {
  constexpr int VPG = Fmt<F>::VPG;
  const int cg = lane / VPG;
  const int s = (int)get_bits(pbytes, f_scale<F>(cg));
  const Bits lo = f_idx_lo<F>(lane);
  const int idx = (int)(get_bits(pbytes, lo) | (get_bits(pbytes, f_idx_hi<F>(lane)) << lo.width));
  int sgn = 0, dbit = 0;
  if (!Fmt<F>::IQ1) {
    sgn = (int)get_bits(pbytes, f_sign<F>(lane));
    if (Fmt<F>::PAR) sgn |= parity7(sgn) << 7;
  } else {
    dbit = F == IQ1_S ? (int)get_bits(pbytes, f_dbit_grp<F>(cg)) : (int)get_bits(pbytes, f_dbit_vec<F>(lane));
  }
  const float *tf = reinterpret_cast<const float *>(tab);
  float g8[8];
#pragma unroll
  for (int i = 0; i < 8; i++) g8[i] = tf[kmaj(idx, i)];
  write_back_vec<F, TIn>(a, b, lane, g8, d, s, sgn, dbit);
}

// Exact rescoring of the flagged items, in one of two layouts chosen by their number.
//
// The choice a block's payload holds for group g (IQ1_S: scale index + delta bit << 3).
template <int F>
__device__ __forceinline__ int payload_choice(const uint8_t *pb, int g) {
  const int c = (int)get_bits(pb, f_scale<F>(g));
  return F == IQ1_S ? c | (int)get_bits(pb, f_dbit_grp<F>(g)) << 3 : c;
}

// A group of which only some vectors are flagged had no near tie between choices, since the sweep
// flags every vector of a group whose choice is near-tied: its choice, which the payload holds, is
// exact, and only its flagged vectors are re-decided under that choice, as with fixed choices.

// CTA per item (used when the items are fewer than the resident warps): one CTA of 4 warps
// re-decides one flagged item at a time, and 4 CTAs share an SM, so that the latency-bound items
// overlap.  Per flagged group, the n vectors it re-decides (all, or with its choice known only the
// flagged ones) share the warps, each over 4 / n slices of the codebook, for the fp32 minima; the
// (near choice, vector, slice) units go to the warps in turn for the fp32 screen of the exact
// minima.  The screen lists its survivors in shared memory and the CTA evaluates the list in fp64
// at once, one thread per candidate: fp64 issues at a small fraction of the fp32 rate on this
// part, so the evaluations are packed into as few warp instructions as possible.  Every reduction
// (a minimum; the least exact error, lowest key on equal errors) gives the same value in any
// order, so the result does not depend on the split.
constexpr int kRsWarps = 4;
constexpr int kRsCtasPerSm = 4;  // 128 registers a thread
constexpr int kRsCap = kRsWarps * 32;  // listed candidates per group: one per thread
constexpr unsigned long long kInfBits = 0x7ff0000000000000ull;  // +inf as a double's bits
struct RescoreSmem {
  uint32_t pay[24];                  // the item's payload bytes
  float part[kRsWarps][16];          // (a) per-warp minima over its slice, per choice
  float mh[4][16];                   // (a) per-vector minima
  double pex[16][4][4];              // (c) long lists: least exact error per (choice, vector, slice)
  int pkey[16][4][4];                //     and its key
  unsigned long long exb[4][16];     // (c) least exact error per (vector, choice), as its bits
  int exkey[4][16];                  //     and its key
  uint32_t cand[kRsCap];             // (c) listed candidates: choice | vector << 4 | key << 8
  float4 candg[kRsCap][2];           //     and their codebook values
  int ncand;
  int nextit;                        // the CTA's next item
};

template <int F, int MODE, typename TIn>
__device__ __forceinline__ void rescore_by_cta(const EncArgs &a, const EncWs &ws, int nflag, RescoreSmem &sm) {
  constexpr int C = Fmt<F>::C, N = Fmt<F>::N, VPG = Fmt<F>::VPG, BB = Fmt<F>::BB, G = Fmt<F>::G;
  static_assert(kRsWarps == 4 && VPG <= 4 && (N / kRsWarps) % 32 == 0, "slices of whole warps");
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const float4 *tab = ws.tab;
  // an item is (block, flagged vectors); every-choice payloads: (block | choice << 27, flagged
  // vectors), re-decided as a fixed-choice block in that choice's payload
  constexpr bool kFixedLike = MODE == MODE_FIXED || MODE == MODE_EVERY;
  uint8_t *pbytes = reinterpret_cast<uint8_t *>(sm.pay);
  // each CTA's first item by its index, every later one from a counter, so that the CTAs whose
  // items were cheap take more
  for (int it = blockIdx.x; it < nflag;) {
    const uint2 item = ws.fb[it];
    const int cpass = MODE == MODE_EVERY ? (int)(item.x >> 27) : 0;
    const int64_t b = MODE == MODE_EVERY ? (int64_t)(item.x & ((1u << 27) - 1u)) : (int64_t)item.x;
    const uint32_t mask = item.y;
    uint8_t *payb = a.payload + (MODE == MODE_EVERY ? (size_t)cpass * a.nblocks * BB : 0) + b * BB;
    for (int i = threadIdx.x; i < BB; i += blockDim.x) pbytes[i] = payb[i];
    Vec v;
    load_block_vec<TIn>(a, b, lane, v);  // every warp holds the whole block
    __syncthreads();
    uint32_t d16;
    if (F == IQ1_M) {
      d16 = 0;
      for (int k = 0; k < 4; k++) d16 |= get_bits(pbytes, f_d16_nib<F>(k)) << (4 * k);
    } else {
      d16 = get_bits(pbytes, f_d16<F>());
    }
    const float d = half_bits_to_float((uint16_t)d16);
    vec_setup<F>(v);
    for (int g = 0; g < G; g++) {
      const uint32_t gm = ((1u << VPG) - 1u) << (g * VPG);
      if (!(mask & gm)) continue;
      const bool fx = kFixedLike || (mask & gm) != gm;  // the group's choice is known
      const int cfix = MODE == MODE_FIXED ? fixed_choice<G>(a, b, g) : MODE == MODE_EVERY ? cpass
                       : fx ? payload_choice<F>(pbytes, g) : -1;
      float Cg = 0.0f;  // the group's sum of w t^2, in vector order (every thread alike)
      for (int k = 0; k < VPG; k++) {
        const float cs = __shfl_sync(0xffffffffu, v.Cs, g * VPG + k);
        Cg = k == 0 ? cs : __fadd_rn(Cg, cs);
      }
      // the vectors re-decided (with the group's choice known only the flagged ones: the entries of
      // the others are independent decisions the sweep already made exactly), each over nsl slices
      // of sl entries
      const uint32_t act = fx ? (mask >> (g * VPG)) & ((1u << VPG) - 1u) : (1u << VPG) - 1u;
      const int nact = __popc(act), nsl = kRsWarps / nact, sl = N / nsl;
      auto act_vec = [&](int r) {  // the r-th re-decided vector of the group
        uint32_t rest = act;
        for (int q = 0; q < r; q++) rest &= rest - 1u;
        return __ffs(rest) - 1;
      };
      // (a) fp32 minima of vector kv over slice js for every choice (or the known one), as the
      // sweep computes them
      const bool kvflag = wid < nact * nsl;
      const int kv = kvflag ? act_vec(wid / nsl) : 0, js = wid % nsl;
      {
        const Vec u = shfl_vec(v, g * VPG + kv);
        float lm[C], alc[C];
#pragma unroll
        for (int c = 0; c < C; c++) {
          lm[c] = INFINITY;
          int s, db0, db1;
          cand_of_choice<F>(c, s, db0, db1);
          alc[c] = alpha_of<F>(d, s);
        }
#pragma unroll 4
        for (int e = js * sl + lane; kvflag && e < (js + 1) * sl; e += 32) {
          Entry en;
          load_entry<F>(a.grid, e, en);
          // the entry's sums once, then every choice's score as cand_score forms it
          float An = 0.0f, Bs = 0.0f, Anp = 0.0f, Bp = 0.0f, Anm = 0.0f, Bm = 0.0f;
          if (!Fmt<F>::IQ1) ab2(u.nw2, u.w, en, An, Bs);
          else ab1(u, en, Anp, Bp, Anm, Bm);
#pragma unroll
          for (int c = 0; c < C; c++) {
            if (fx && c != cfix) continue;
            int s, db0, db1;
            cand_of_choice<F>(c, s, db0, db1);
            if (!Fmt<F>::IQ1) {
              lm[c] = fminf(lm[c], __fmaf_rn(alc[c], Bs, An));
            } else {
              lm[c] = fminf(lm[c], db0 ? __fmaf_rn(alc[c], Bm, Anm) : __fmaf_rn(alc[c], Bp, Anp));
              if (db1 != db0) lm[c] = fminf(lm[c], db1 ? __fmaf_rn(alc[c], Bm, Anm) : __fmaf_rn(alc[c], Bp, Anp));
            }
          }
        }
#pragma unroll
        for (int c = 0; c < C; c++) {
          float x = lm[c];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) x = fminf(x, __shfl_xor_sync(0xffffffffu, x, off));
          if (lane == 0) sm.part[wid][c] = x;
        }
      }
      __syncthreads();
      for (int t = threadIdx.x; t < VPG * C; t += blockDim.x) {
        const int k = t / C, c = t % C;
        float x = INFINITY;
        if ((act >> k) & 1u) {
          const int r = __popc(act & ((1u << k) - 1u));
          for (int j = 0; j < nsl; j++) x = fminf(x, sm.part[r * nsl + j][c]);
        }
        sm.mh[k][c] = x;
        sm.exb[k][c] = kInfBits;
        sm.exkey[k][c] = 0x7fffffff;
      }
      if (threadIdx.x == 0) sm.ncand = 0;
      __syncthreads();
      // (b) near set of choices (every thread alike)
      uint32_t near = 0;
      {
        float D[C];
        float D1 = INFINITY;
        for (int c = 0; c < C; c++) {
          if (fx && c != cfix) { D[c] = INFINITY; continue; }
          float S = sm.mh[0][c];
          for (int k = 1; k < VPG; k++) S = __fadd_rn(S, sm.mh[k][c]);
          D[c] = __fmul_rn(alpha_choice<F>(d, c), S);
          D1 = fminf(D1, D[c]);
        }
        for (int c = 0; c < C; c++)
          if (D[c] != INFINITY && __fsub_rn(D[c], D1) <= kMargin * (4.0f * Cg + D1 + D[c])) near |= 1u << c;
        if (fx) near = 1u << cfix;
      }
      // (c) exact minimum per (near choice, vector) over the candidates the bound cannot exclude:
      // units (near choice, vector, slice) dealt to the warps screen in fp32.  LISTED: the
      // survivors go to the shared list; otherwise (a list longer than its capacity: many
      // candidates within the bound) each unit evaluates its own survivors in fp64.
      const int nunits = __popc(near) * nact * nsl;
      auto run_units = [&](auto listed_t) {
        constexpr bool LISTED = decltype(listed_t)::value;
        for (int unit = wid; unit < nunits; unit += kRsWarps) {
          const int ci = unit / (nact * nsl), k = act_vec((unit / nsl) % nact), j = unit % nsl;
          uint32_t rest = near;
          for (int q = 0; q < ci; q++) rest &= rest - 1u;
          const int c = __ffs(rest) - 1;
          int s, db0, db1;
          cand_of_choice<F>(c, s, db0, db1);
          const float al = alpha_of<F>(d, s);
          const Vec u = shfl_vec(v, g * VPG + k);
          const float emin = __fmul_rn(al, sm.mh[k][c]);
          double bestE = INFINITY;
          int bestK = 0x7fffffff;
#pragma unroll 4
          for (int e = j * sl + lane; e < (j + 1) * sl; e += 32) {  // the same trip count in every lane
            Entry en;
            load_entry<F>(a.grid, e, en);
            for (int db = db0; db <= db1; db++) {
              const float sc = cand_score<F>(u, en, al, db);
              const float ec = __fmul_rn(al, sc);
              const bool pass = __fsub_rn(ec, emin) <= kMargin * (4.0f * u.Cs + emin + ec);
              const int kk = (F == IQ1_M ? db * N : 0) + e;
              if constexpr (LISTED) {
                const uint32_t pm = __ballot_sync(0xffffffffu, pass);
                if (pm) {
                  int base = 0;
                  if (lane == 0) base = atomicAdd(&sm.ncand, __popc(pm));
                  base = __shfl_sync(0xffffffffu, base, 0);
                  const int slot = base + __popc(pm & ((1u << lane) - 1u));
                  if (pass && slot < kRsCap) {
                    sm.cand[slot] = (uint32_t)c | ((uint32_t)k << 4) | ((uint32_t)kk << 8);
                    sm.candg[slot][0] = make_float4(en.g[0], en.g[1], en.g[2], en.g[3]);
                    sm.candg[slot][1] = make_float4(en.g[4], en.g[5], en.g[6], en.g[7]);
                  }
                }
              } else if (pass) {
                const double E = exact_err<F>(u.x, u.w, en, d, s, u.sgn, db);
                if (E < bestE || (E == bestE && kk < bestK)) { bestE = E; bestK = kk; }
              }
            }
          }
          if constexpr (!LISTED) {
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
              const double oE = __shfl_xor_sync(0xffffffffu, bestE, off);
              const int oK = __shfl_xor_sync(0xffffffffu, bestK, off);
              if (oE < bestE || (oE == bestE && oK < bestK)) { bestE = oE; bestK = oK; }
            }
            if (lane == 0) { sm.pex[c][k][j] = bestE; sm.pkey[c][k][j] = bestK; }
          }
        }
      };
      run_units(std::true_type{});
      __syncthreads();
      const int ncand = sm.ncand;
      if (ncand <= kRsCap) {
        // one listed candidate per thread; the exact error E >= +0 (non-negative weights), so the
        // least error is the least bit pattern, and the lowest key is taken among the equal ones
        const int i = threadIdx.x;
        const uint32_t cd = i < ncand ? sm.cand[i] : 0u;
        const int c = cd & 15u, k = (cd >> 4) & 15u, kk = (int)(cd >> 8);
        const Vec u = shfl_vec(v, g * VPG + k);
        unsigned long long eb = 0;
        if (i < ncand) {
          int s, db0, db1;
          cand_of_choice<F>(c, s, db0, db1);
          Entry en;  // the codebook values the screen kept (the direct form reads only g)
          const float4 g0 = sm.candg[i][0], g1 = sm.candg[i][1];
          en.g[0] = g0.x; en.g[1] = g0.y; en.g[2] = g0.z; en.g[3] = g0.w;
          en.g[4] = g1.x; en.g[5] = g1.y; en.g[6] = g1.z; en.g[7] = g1.w;
          eb = (unsigned long long)__double_as_longlong(exact_err<F>(u.x, u.w, en, d, s, u.sgn, F == IQ1_M ? kk / N : db0));
          atomicMin(&sm.exb[k][c], eb);
        }
        __syncthreads();
        if (i < ncand && eb == sm.exb[k][c]) atomicMin(&sm.exkey[k][c], kk);
      } else {
        run_units(std::false_type{});
        __syncthreads();
        for (int t = threadIdx.x; t < VPG * C; t += blockDim.x) {
          const int k = t / C, c = t % C;
          if (!((near >> c) & 1) || !((act >> k) & 1u)) continue;
          double E = sm.pex[c][k][0];
          int K = sm.pkey[c][k][0];
          for (int j = 1; j < nsl; j++) {
            const double oE = sm.pex[c][k][j];
            const int oK = sm.pkey[c][k][j];
            if (oE < E || (oE == E && oK < K)) { E = oE; K = oK; }
          }
          sm.exb[k][c] = (unsigned long long)__double_as_longlong(E);
          sm.exkey[k][c] = K;
        }
      }
      __syncthreads();
      // (d) exact choice: least sum over the vectors, lowest choice on equal error; (e) rewrite the
      // group's fields (keep the sweep's decision if nothing was comparable)
      if (threadIdx.x == 0) {
        const bool one = __popc(near) == 1;  // a single near choice needs no sums
        int cstar = one ? __ffs(near) - 1 : -1;
        double bestG = INFINITY;
        for (int c = 0; !one && c < C; c++) {
          if (!((near >> c) & 1)) continue;
          double Eg = __longlong_as_double((long long)sm.exb[0][c]);
          for (int k = 1; k < VPG; k++) Eg = __dadd_rn(Eg, __longlong_as_double((long long)sm.exb[k][c]));
          if (cstar < 0 || Eg < bestG) { bestG = Eg; cstar = c; }
        }
        if (fx) cstar = cfix;
        if (cstar >= 0) {
          set_bits_bytes(pbytes, f_scale<F>(g), (uint32_t)(F == IQ1_S ? (cstar & 7) : cstar));
          if (F == IQ1_S) set_bits_bytes(pbytes, f_dbit_grp<F>(g), (uint32_t)(cstar >> 3));
          for (int k = 0; k < VPG; k++) {
            const int vv = g * VPG + k;
            if (fx && !((mask >> vv) & 1u)) continue;
            const int key = sm.exkey[k][cstar];
            const int idx = F == IQ1_M ? key % N : key;
            const Bits lo = f_idx_lo<F>(vv);
            set_bits_bytes(pbytes, lo, (uint32_t)idx);
            if (F == IQ2_S || Fmt<F>::IQ1) set_bits_bytes(pbytes, f_idx_hi<F>(vv), (uint32_t)idx >> lo.width);
            if (F == IQ1_M) set_bits_bytes(pbytes, f_dbit_vec<F>(vv), (uint32_t)(key / N));
          }
        }
      }
      __syncthreads();
    }
    for (int i = threadIdx.x; i < BB; i += blockDim.x) payb[i] = pbytes[i];
    if (a.wb && wid == 0) write_back_bytes<F, TIn>(a, tab, b, lane, pbytes, d);
    if (threadIdx.x == 0) sm.nextit = (int)gridDim.x + atomicAdd(&ws.hdr[2], 1);
    __syncthreads();  // the payload bytes are reused by the next item
    it = sm.nextit;
  }
}

constexpr int kRsWarpCap = 64;  // listed candidates per group, warp per item
struct RescoreWarpSmem {
  float mh[4][16];
  unsigned long long exb[4][16];     // least exact error per (vector, choice), as its bits
  int exkey[4][16];                  // and its key
  uint32_t cand[kRsWarpCap];         // listed candidates: choice | vector << 4 | key << 8
  float4 candg[kRsWarpCap][2];       // and their codebook values
  unsigned long long ceb[kRsWarpCap];  // their exact errors' bits
  uint32_t pay[24];
};

// Warp per item: each warp re-decides its own items, so that the warps' load latencies overlap
// (used when the items outnumber the resident warps).
template <int F, int MODE, typename TIn>
__device__ __forceinline__ void rescore_by_warp(const EncArgs &a, const EncWs &ws, int nflag, RescoreWarpSmem &sm) {
  constexpr int C = Fmt<F>::C, N = Fmt<F>::N, VPG = Fmt<F>::VPG, BB = Fmt<F>::BB, G = Fmt<F>::G;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const float4 *tab = ws.tab;
  // an item is (block, flagged vectors); every-choice payloads: (block | choice << 27, flagged
  // vectors), re-decided as a fixed-choice block in that choice's payload
  constexpr bool kFixedLike = MODE == MODE_FIXED || MODE == MODE_EVERY;
  // each warp's first item by its index, every later one from a counter
  for (int it = blockIdx.x * kRsWarps + wid; it < nflag;) {
   const uint2 item = ws.fb[it];
   {
    const int cpass = MODE == MODE_EVERY ? (int)(item.x >> 27) : 0;
    const int64_t b = MODE == MODE_EVERY ? (int64_t)(item.x & ((1u << 27) - 1u)) : (int64_t)item.x;
    const uint32_t mask = item.y;
    uint8_t *payb = a.payload + (MODE == MODE_EVERY ? (size_t)cpass * a.nblocks * BB : 0) + b * BB;
    Vec v;
    load_block_vec<TIn>(a, b, lane, v);
    uint8_t *pbytes = reinterpret_cast<uint8_t *>(sm.pay);
    for (int i = lane; i < BB; i += 32) pbytes[i] = payb[i];
    __syncwarp();
    uint32_t d16;
    if (F == IQ1_M) {
      d16 = 0;
      for (int k = 0; k < 4; k++) d16 |= get_bits(pbytes, f_d16_nib<F>(k)) << (4 * k);
    } else {
      d16 = get_bits(pbytes, f_d16<F>());
    }
    __syncwarp();
    const float d = half_bits_to_float((uint16_t)d16);
    vec_setup<F>(v);
    for (int g = 0; g < G; g++) {
      const uint32_t gm = ((1u << VPG) - 1u) << (g * VPG);
      if (!(mask & gm)) continue;
      float Cg = 0.0f;
      // (a) fp32 per-vector minima for every choice (or the known one), as the sweep computes them.
      // With the group's choice known, the vectors' entries are independent decisions: only the
      // flagged vectors are re-decided, the others keep the sweep's exact pick.
      const bool fx = kFixedLike || (mask & gm) != gm;
      const int cfix = MODE == MODE_FIXED ? fixed_choice<G>(a, b, g) : MODE == MODE_EVERY ? cpass
                       : fx ? payload_choice<F>(pbytes, g) : -1;
      for (int k = 0; k < VPG; k++) {
        const Vec u = shfl_vec(v, g * VPG + k);
        Cg = k == 0 ? u.Cs : __fadd_rn(Cg, u.Cs);
        if (fx && !((mask >> (g * VPG + k)) & 1u)) continue;
        float lm[C], alc[C];
#pragma unroll
        for (int c = 0; c < C; c++) {
          lm[c] = INFINITY;
          int s, db0, db1;
          cand_of_choice<F>(c, s, db0, db1);
          alc[c] = alpha_of<F>(d, s);
        }
#pragma unroll 4
        for (int e = lane; e < N; e += 32) {
          Entry en;
          load_entry<F>(a.grid, e, en);
          // the entry's sums once, then every choice's score as cand_score forms it
          float An = 0.0f, Bs = 0.0f, Anp = 0.0f, Bp = 0.0f, Anm = 0.0f, Bm = 0.0f;
          if (!Fmt<F>::IQ1) ab2(u.nw2, u.w, en, An, Bs);
          else ab1(u, en, Anp, Bp, Anm, Bm);
#pragma unroll
          for (int c = 0; c < C; c++) {
            if (fx && c != cfix) continue;
            int s, db0, db1;
            cand_of_choice<F>(c, s, db0, db1);
            if (!Fmt<F>::IQ1) {
              lm[c] = fminf(lm[c], __fmaf_rn(alc[c], Bs, An));
            } else {
              lm[c] = fminf(lm[c], db0 ? __fmaf_rn(alc[c], Bm, Anm) : __fmaf_rn(alc[c], Bp, Anp));
              if (db1 != db0) lm[c] = fminf(lm[c], db1 ? __fmaf_rn(alc[c], Bm, Anm) : __fmaf_rn(alc[c], Bp, Anp));
            }
          }
        }
#pragma unroll
        for (int c = 0; c < C; c++) {
          float x = lm[c];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) x = fminf(x, __shfl_xor_sync(0xffffffffu, x, off));
          lm[c] = x;
        }
        if (lane == 0)
          for (int c = 0; c < C; c++) sm.mh[k][c] = lm[c];
      }
      __syncwarp();
      // (b) near set of choices
      float D[C];
      float D1 = INFINITY;
      for (int c = 0; c < C; c++) {
        if (fx && c != cfix) { D[c] = INFINITY; continue; }
        float S = sm.mh[0][c];
        for (int k = 1; k < VPG; k++) S = __fadd_rn(S, sm.mh[k][c]);
        D[c] = __fmul_rn(alpha_choice<F>(d, c), S);
        D1 = fminf(D1, D[c]);
      }
      uint32_t near = 0;
      for (int c = 0; c < C; c++)
        if (D[c] != INFINITY && __fsub_rn(D[c], D1) <= kMargin * (4.0f * Cg + D1 + D[c])) near |= 1u << c;
      if (fx) near = 1u << cfix;
      // (c) exact minimum per (vector, near choice) over the candidates the bound cannot exclude:
      // the fp32 screen lists its survivors and the warp evaluates the list in fp64 together, one
      // lane per candidate; the least error is the least bit pattern (E >= +0), the lowest key is
      // taken among the equal ones.  A list longer than its capacity: each (vector, choice) in turn.
      for (int t = lane; t < VPG * C; t += 32) { sm.exb[t / C][t % C] = kInfBits; sm.exkey[t / C][t % C] = 0x7fffffff; }
      __syncwarp();
      auto run_pairs = [&](auto listed_t) -> int {
        constexpr bool LISTED = decltype(listed_t)::value;
        int ncand = 0;
        for (int c = 0; c < C; c++) {
          if (!((near >> c) & 1)) continue;
          int s, db0, db1;
          cand_of_choice<F>(c, s, db0, db1);
          const float al = alpha_of<F>(d, s);
          for (int k = 0; k < VPG; k++) {
            if (fx && !((mask >> (g * VPG + k)) & 1u)) continue;
            const Vec u = shfl_vec(v, g * VPG + k);
            const float emin = __fmul_rn(al, sm.mh[k][c]);
            double bestE = INFINITY;
            int bestK = 0x7fffffff;
#pragma unroll 4
            for (int e = lane; e < N; e += 32) {  // the same trip count in every lane
              Entry en;
              load_entry<F>(a.grid, e, en);
              for (int db = db0; db <= db1; db++) {
                const float sc = cand_score<F>(u, en, al, db);
                const float ec = __fmul_rn(al, sc);
                const bool pass = __fsub_rn(ec, emin) <= kMargin * (4.0f * u.Cs + emin + ec);
                const int kk = (F == IQ1_M ? db * N : 0) + e;
                if constexpr (LISTED) {
                  const uint32_t pm = __ballot_sync(0xffffffffu, pass);
                  const int slot = ncand + __popc(pm & ((1u << lane) - 1u));
                  if (pass && slot < kRsWarpCap) {
                    sm.cand[slot] = (uint32_t)c | ((uint32_t)k << 4) | ((uint32_t)kk << 8);
                    sm.candg[slot][0] = make_float4(en.g[0], en.g[1], en.g[2], en.g[3]);
                    sm.candg[slot][1] = make_float4(en.g[4], en.g[5], en.g[6], en.g[7]);
                  }
                  ncand += __popc(pm);
                } else if (pass) {
                  const double E = exact_err<F>(u.x, u.w, en, d, s, u.sgn, db);
                  if (E < bestE || (E == bestE && kk < bestK)) { bestE = E; bestK = kk; }
                }
              }
            }
            if constexpr (!LISTED) {
#pragma unroll
              for (int off = 16; off >= 1; off >>= 1) {
                const double oE = __shfl_xor_sync(0xffffffffu, bestE, off);
                const int oK = __shfl_xor_sync(0xffffffffu, bestK, off);
                if (oE < bestE || (oE == bestE && oK < bestK)) { bestE = oE; bestK = oK; }
              }
              if (lane == 0) { sm.exb[k][c] = (unsigned long long)__double_as_longlong(bestE); sm.exkey[k][c] = bestK; }
            }
          }
        }
        return ncand;
      };
      const int ncand = run_pairs(std::true_type{});
      __syncwarp();
      if (ncand <= kRsWarpCap) {
        for (int i0 = 0; i0 < ncand; i0 += 32) {  // the same trip count in every lane
          const int i = i0 + lane;
          const uint32_t cd = i < ncand ? sm.cand[i] : 0u;
          const int c = cd & 15u, k = (cd >> 4) & 15u, kk = (int)(cd >> 8);
          const Vec u = shfl_vec(v, g * VPG + k);
          if (i < ncand) {
            int s, db0, db1;
            cand_of_choice<F>(c, s, db0, db1);
            Entry en;  // the codebook values the screen kept (the direct form reads only g)
            const float4 g0 = sm.candg[i][0], g1 = sm.candg[i][1];
            en.g[0] = g0.x; en.g[1] = g0.y; en.g[2] = g0.z; en.g[3] = g0.w;
            en.g[4] = g1.x; en.g[5] = g1.y; en.g[6] = g1.z; en.g[7] = g1.w;
            const unsigned long long eb =
                (unsigned long long)__double_as_longlong(exact_err<F>(u.x, u.w, en, d, s, u.sgn, F == IQ1_M ? kk / N : db0));
            sm.ceb[i] = eb;
            atomicMin(&sm.exb[k][c], eb);
          }
        }
        __syncwarp();
        for (int i = lane; i < ncand; i += 32) {
          const uint32_t cd = sm.cand[i];
          const int c = cd & 15u, k = (cd >> 4) & 15u;
          if (sm.ceb[i] == sm.exb[k][c]) atomicMin(&sm.exkey[k][c], (int)(cd >> 8));
        }
      } else {
        run_pairs(std::false_type{});
      }
      __syncwarp();
      // (d) exact choice: least sum over the vectors, lowest choice on equal error
      const bool one = __popc(near) == 1;  // a single near choice needs no sums
      int cstar = one ? __ffs(near) - 1 : -1;
      double bestG = INFINITY;
      for (int c = 0; !one && c < C; c++) {
        if (!((near >> c) & 1)) continue;
        double Eg = __longlong_as_double((long long)sm.exb[0][c]);
        for (int k = 1; k < VPG; k++) Eg = __dadd_rn(Eg, __longlong_as_double((long long)sm.exb[k][c]));
        if (cstar < 0 || Eg < bestG) { bestG = Eg; cstar = c; }
      }
      if (fx) cstar = cfix;
      // (e) rewrite the group's fields (keep the sweep's decision if nothing was comparable)
      if (lane == 0 && cstar >= 0) {
        set_bits_bytes(pbytes, f_scale<F>(g), (uint32_t)(F == IQ1_S ? (cstar & 7) : cstar));
        if (F == IQ1_S) set_bits_bytes(pbytes, f_dbit_grp<F>(g), (uint32_t)(cstar >> 3));
        for (int k = 0; k < VPG; k++) {
          const int vv = g * VPG + k;
          if (fx && !((mask >> vv) & 1u)) continue;
          const int key = sm.exkey[k][cstar];
          const int idx = F == IQ1_M ? key % N : key;
          const Bits lo = f_idx_lo<F>(vv);
          set_bits_bytes(pbytes, lo, (uint32_t)idx);
          if (F == IQ2_S || Fmt<F>::IQ1) set_bits_bytes(pbytes, f_idx_hi<F>(vv), (uint32_t)idx >> lo.width);
          if (F == IQ1_M) set_bits_bytes(pbytes, f_dbit_vec<F>(vv), (uint32_t)(key / N));
        }
      }
      __syncwarp();
    }
    for (int i = lane; i < BB; i += 32) payb[i] = pbytes[i];
    if (a.wb) write_back_bytes<F, TIn>(a, tab, b, lane, pbytes, d);
    __syncwarp();
   }
   int nx = 0;
   if (lane == 0) nx = (int)gridDim.x * kRsWarps + atomicAdd(&ws.hdr[2], 1);
   it = __shfl_sync(0xffffffffu, nx, 0);
  }
}

template <int F, int MODE, typename TIn>
__global__ void __launch_bounds__(kRsWarps * 32, kRsCtasPerSm) rescore_kernel(EncArgs a, EncWs ws) {
  __shared__ RescoreSmem sm;
  __shared__ RescoreWarpSmem smw[kRsWarps];
  const int nflag = ws.hdr[1];  // the same for every CTA, so every CTA takes the same layout
  if (nflag >= kRsWarps * (int)gridDim.x) rescore_by_warp<F, MODE, TIn>(a, ws, nflag, smw[threadIdx.x >> 5]);
  else rescore_by_cta<F, MODE, TIn>(a, ws, nflag, sm);
}

// ---------------------------------------------------------------------------------------------
template <int F, typename TIn>
__global__ void __launch_bounds__(256) anchor_kernel(const TIn *__restrict__ W, int64_t cols, int64_t nblocks,
                                                     uint16_t *__restrict__ d16, int32_t *__restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t bpr = cols / 256;
  int st = 0;
  for (int64_t b = warp; b < nblocks; b += nw) {
    float x[8];
    load8(W + (b / bpr) * cols + (b % bpr) * 256 + lane * 8, x);
    const bool fin = __all_sync(0xffffffffu, finite8(x));
    uint16_t h = 0;
    if (fin) h = half_bits_rn(anchor_scale<F>(x));
    else st |= IQ_STATUS_BAD_INPUT;
    if (lane == 0) d16[b] = h;
  }
  if (st && lane == 0 && status) atomicOr(status, st);
}

static int num_sms() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

template <int F, typename TIn>
static int run_anchor(const void *W, int64_t cols, int64_t nb, uint16_t *d16, int32_t *status, cudaStream_t st) {
  if (nb == 0) return IQ_OK;
  const int64_t want = (nb + 7) / 8;
  const int grid = (int)(want < (int64_t)num_sms() * 8 ? want : (int64_t)num_sms() * 8);
  anchor_kernel<F, TIn><<<grid, 256, 0, st>>>((const TIn *)W, cols, nb, d16, status);
  return cudaPeekAtLastError() == cudaSuccess ? IQ_OK : IQ_ERR_CUDA;
}

template <int F, int MODE, typename TIn>
static int run_encode(const EncArgs &a, void *workspace, size_t ws_bytes, cudaStream_t st) {
  constexpr int N = Fmt<F>::N;
  if (a.nblocks == 0) return IQ_OK;
  EncWs ws = enc_ws(workspace, N);
  if (cudaMemsetAsync(ws.hdr, 0, 256, st) != cudaSuccess) return IQ_ERR_CUDA;
  prep_codebook<F><<<(N + 255) / 256, 256, 0, st>>>(a.grid, ws);
  const size_t smem = tc_smem<F, MODE>(tc_nbuf<F, MODE>());
  auto kern = encode_tc_kernel<F, MODE, TIn>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return IQ_ERR_CUDA;
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTcThreads, smem);
  if (per_sm < 1) per_sm = 1;
  // tensor memory: at most 512 columns per SM among the resident CTAs
  if (per_sm * TcCfg<F>::ALLOC > 512) per_sm = 512 / TcCfg<F>::ALLOC;
  const int64_t nquads = (a.nblocks + 3) / 4;
  const int64_t cap = (int64_t)num_sms() * per_sm;
  const int grid = (int)(nquads < cap ? nquads : cap);
  kern<<<grid, kTcThreads, smem, st>>>(a, ws, nquads);
  if (cudaPeekAtLastError() != cudaSuccess) return IQ_ERR_CUDA;
  if (MODE != MODE_TABLE) {
    auto rk = rescore_kernel<F, MODE, TIn>;
    int rs_per_sm = 2;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&rs_per_sm, rk, kRsWarps * 32, 0);
    rk<<<num_sms() * (rs_per_sm > 1 ? rs_per_sm : 1), kRsWarps * 32, 0, st>>>(a, ws);
    if (cudaPeekAtLastError() != cudaSuccess) return IQ_ERR_CUDA;
  }
  return IQ_OK;
}

template <int MODE, typename TIn>
static int dispatch_encode(iq_format f, const EncArgs &a, void *ws, size_t wsb, cudaStream_t st) {
  switch (f) {
    case IQ2_XXS: return run_encode<IQ2_XXS, MODE, TIn>(a, ws, wsb, st);
    case IQ2_XS: return run_encode<IQ2_XS, MODE, TIn>(a, ws, wsb, st);
    case IQ2_S: return run_encode<IQ2_S, MODE, TIn>(a, ws, wsb, st);
    case IQ1_S: return run_encode<IQ1_S, MODE, TIn>(a, ws, wsb, st);
    default: return run_encode<IQ1_M, MODE, TIn>(a, ws, wsb, st);
  }
}

static int grid_entries(iq_format f) {
  return f == IQ2_XXS ? 256 : f == IQ2_XS ? 512 : f == IQ2_S ? 1024 : 2048;
}

static int check_common(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols, const float *imp,
                        int64_t rpe, const float *grid) {
  if ((unsigned)f > IQ1_M || (dt != IQ_F32 && dt != IQ_BF16)) return IQ_ERR_ARG;
  if (rows < 0 || cols <= 0 || cols % 256) return IQ_ERR_ARG;
  if (rows * (cols / 256) >= (int64_t)1 << 32) return IQ_ERR_ARG;
  if (rpe < 0 || (rpe > 0 && rows % rpe)) return IQ_ERR_ARG;
  if (rows > 0 && (!W || !grid)) return IQ_ERR_ARG;
  if (((uintptr_t)W & 15) || ((uintptr_t)grid & 15) || ((uintptr_t)imp & 15)) return IQ_ERR_ARG;
  return IQ_OK;
}

}  // namespace iqk

using namespace iqk;

extern "C" int iq_anchor_scales(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols, uint16_t *d16,
                                int32_t *status, void *stream) {
  if ((unsigned)f > IQ1_M || (dt != IQ_F32 && dt != IQ_BF16) || rows < 0 || cols <= 0 || cols % 256) return IQ_ERR_ARG;
  const int64_t nb = rows * (cols / 256);
  if (nb > 0 && (!W || !d16)) return IQ_ERR_ARG;
  if ((uintptr_t)W & 15) return IQ_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
#define IQ_ANCHOR_CASE(FF)                                                                  \
  case FF:                                                                                  \
    return dt == IQ_BF16 ? run_anchor<FF, __nv_bfloat16>(W, cols, nb, d16, status, st)      \
                         : run_anchor<FF, float>(W, cols, nb, d16, status, st);
  switch (f) {
    IQ_ANCHOR_CASE(IQ2_XXS)
    IQ_ANCHOR_CASE(IQ2_XS)
    IQ_ANCHOR_CASE(IQ2_S)
    IQ_ANCHOR_CASE(IQ1_S)
    IQ_ANCHOR_CASE(IQ1_M)
  }
#undef IQ_ANCHOR_CASE
  return IQ_ERR_ARG;
}

extern "C" int iq_encode_workspace_size(iq_format f, int64_t rows, int64_t cols, size_t *bytes) {
  if ((unsigned)f > IQ1_M || rows < 0 || cols <= 0 || cols % 256 || !bytes) return IQ_ERR_ARG;
  *bytes = enc_ws_bytes(grid_entries(f), rows * (cols / 256));
  return IQ_OK;
}

extern "C" int iq_encode(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols, const float *importance,
                         int64_t rows_per_expert, const float *grid, const uint16_t *d16, const uint8_t *choices,
                         uint8_t *payload, float *group_errors, int32_t *status, void *workspace,
                         size_t workspace_bytes, void *stream) {
  int rc = check_common(f, W, dt, rows, cols, importance, rows_per_expert, grid);
  if (rc) return rc;
  const int64_t nb = rows * (cols / 256);
  if (nb > 0 && !payload) return IQ_ERR_ARG;
  if (choices && group_errors) return IQ_ERR_ARG;  // the table is a product of the search
  if ((uintptr_t)group_errors & 15) return IQ_ERR_ARG;
  size_t need = 0;
  iq_encode_workspace_size(f, rows, cols, &need);
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255)) return IQ_ERR_WORKSPACE;
  EncArgs a{W, rows, cols, nb, importance, rows_per_expert, grid, d16, choices, payload, group_errors, status, 0, nullptr};
  cudaStream_t st = (cudaStream_t)stream;
  if (choices)
    return dt == IQ_BF16 ? dispatch_encode<MODE_FIXED, __nv_bfloat16>(f, a, workspace, workspace_bytes, st)
                         : dispatch_encode<MODE_FIXED, float>(f, a, workspace, workspace_bytes, st);
  return dt == IQ_BF16 ? dispatch_encode<MODE_SEARCH, __nv_bfloat16>(f, a, workspace, workspace_bytes, st)
                       : dispatch_encode<MODE_SEARCH, float>(f, a, workspace, workspace_bytes, st);
}

// Encode and write the decoded weight back ("Add imatrix calibration for the GGML formats ...",
// What imatrix does: the encoder encodes each weight with its statistic, writes the decoded weight
// back and pins the payload), fused: the encoder writes each block's decoded values over W in its
// epilogue, and the exact rescoring writes the blocks it re-decides after their final decisions,
// so W is read once and the payload is not read back.
extern "C" int iq_encode_write_back(iq_format f, void *W, iq_dtype dt, int64_t rows, int64_t cols,
                                    const float *importance, int64_t rows_per_expert, const float *grid,
                                    const uint16_t *d16, const uint8_t *choices, uint8_t *payload, int32_t *status,
                                    void *workspace, size_t workspace_bytes, void *stream) {
  int rc = check_common(f, W, dt, rows, cols, importance, rows_per_expert, grid);
  if (rc) return rc;
  const int64_t nb = rows * (cols / 256);
  if (nb > 0 && !payload) return IQ_ERR_ARG;
  size_t need = 0;
  iq_encode_workspace_size(f, rows, cols, &need);
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255)) return IQ_ERR_WORKSPACE;
  EncArgs a{W, rows, cols, nb, importance, rows_per_expert, grid, d16, choices, payload, nullptr, status, 0, W};
  cudaStream_t st = (cudaStream_t)stream;
  if (choices)
    return dt == IQ_BF16 ? dispatch_encode<MODE_FIXED, __nv_bfloat16>(f, a, workspace, workspace_bytes, st)
                         : dispatch_encode<MODE_FIXED, float>(f, a, workspace, workspace_bytes, st);
  return dt == IQ_BF16 ? dispatch_encode<MODE_SEARCH, __nv_bfloat16>(f, a, workspace, workspace_bytes, st)
                       : dispatch_encode<MODE_SEARCH, float>(f, a, workspace, workspace_bytes, st);
}

extern "C" int iq_group_errors(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols,
                               const float *importance, int64_t rows_per_expert, const float *grid, const uint16_t *d16,
                               float *group_errors, int32_t *status, void *workspace, size_t workspace_bytes,
                               void *stream) {
  int rc = check_common(f, W, dt, rows, cols, importance, rows_per_expert, grid);
  if (rc) return rc;
  const int64_t nb = rows * (cols / 256);
  if (nb > 0 && !group_errors) return IQ_ERR_ARG;
  if ((uintptr_t)group_errors & 15) return IQ_ERR_ARG;
  size_t need = 0;
  iq_encode_workspace_size(f, rows, cols, &need);
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255)) return IQ_ERR_WORKSPACE;
  EncArgs a{W, rows, cols, nb, importance, rows_per_expert, grid, d16, nullptr, nullptr, group_errors, status, 0, nullptr};
  cudaStream_t st = (cudaStream_t)stream;
  return dt == IQ_BF16 ? dispatch_encode<MODE_TABLE, __nv_bfloat16>(f, a, workspace, workspace_bytes, st)
                       : dispatch_encode<MODE_TABLE, float>(f, a, workspace, workspace_bytes, st);
}

// Every-choice payloads (PR #3159): payload c is the forced encode with every group at choice c,
// from one pass: sweep 1 gives every choice's minimum per vector, sweep 2 the entry that attains it
// under every choice, and near ties are rescored exactly per (block, choice), so every payload is
// byte-identical to the forced encode.
extern "C" int iq_encode_every_choice(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols,
                                      const float *importance, int64_t rows_per_expert, const float *grid,
                                      const uint16_t *d16, uint8_t *payloads, int32_t *status, void *workspace,
                                      size_t workspace_bytes, void *stream) {
  int rc = check_common(f, W, dt, rows, cols, importance, rows_per_expert, grid);
  if (rc) return rc;
  const int64_t nb = rows * (cols / 256);
  if (nb > 0 && !payloads) return IQ_ERR_ARG;
  if (nb >= ((int64_t)1 << 27)) return IQ_ERR_TOO_LARGE;  // flag items carry the block in 27 bits
  iq_format_info_t info;
  iq_format_info(f, &info);
  size_t need = 0;
  iq_encode_workspace_size(f, rows * info.num_choices, cols, &need);  // a flag list entry per (block, choice)
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255)) return IQ_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  EncArgs a{W, rows, cols, nb, importance, rows_per_expert, grid, d16, nullptr, payloads, nullptr, status, 0, nullptr};
  return dt == IQ_BF16 ? dispatch_encode<MODE_EVERY, __nv_bfloat16>(f, a, workspace, workspace_bytes, st)
                       : dispatch_encode<MODE_EVERY, float>(f, a, workspace, workspace_bytes, st);
}

extern "C" int iq_format_info(iq_format f, iq_format_info_t *out) {
  if ((unsigned)f > IQ1_M || !out) return IQ_ERR_ARG;
  const int bits[5] = {8, 9, 10, 11, 11};
  const int G[5] = {8, 16, 16, 8, 16}, C[5] = {16, 16, 16, 16, 8}, V[5] = {4, 2, 2, 4, 2};
  out->block_bytes = fmt_block_bytes(f);
  out->choice_groups = G[f];
  out->num_choices = C[f];
  out->grid_entries = grid_entries(f);
  out->vectors_per_group = V[f];
  out->index_bits = bits[f];
  return IQ_OK;
}

// ---------------------------------------------------------------------------------------------
// Encoder for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc, or to take memory from a caching allocator:
// code that runs while a stream is being captured into a CUDA graph in the global capture mode
// (where cudaMalloc is refused), plug-ins loaded into a host framework that owns every byte of
// device memory through its own pool, and latency-bound serving loops that may not block on an
// allocation.  They still own their inputs and outputs, but cannot provide the scratch
// `workspace` that iq_encode needs.  This entry point takes its scratch from one file-scope
// device array instead.
//
// The array is kStaticScratchBytes (1 MiB) per GPU, held by every device that loads the library
// until the process exits.  Every call on a device shares it: the header the kernels count in is
// cleared by each call before use, and calls whose kernels overlap on the GPU (for example on two
// streams) race on it, so issue them in order on one stream.
namespace iqk {
constexpr size_t kStaticScratchBytes = (size_t)1 << 20;
static __device__ __align__(256) uint8_t g_encode_scratch[kStaticScratchBytes];

// Device address of g_encode_scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device with cudaGetSymbolAddress
// (the first call on a device does this; make that first call before any stream capture).
static void *static_scratch_ptr() {
  constexpr int kMaxDevices = 64;
  static void *ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_encode_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}
}  // namespace iqk

extern "C" int iq_encode_static_scratch_capacity(iq_format f, int64_t *max_blocks) {
  if ((unsigned)f > IQ1_M || !max_blocks) return IQ_ERR_ARG;
  const size_t fixed = 256 + al256((size_t)grid_entries(f) * 64);
  *max_blocks = (int64_t)((kStaticScratchBytes - fixed) / 8);
  return IQ_OK;
}

extern "C" int iq_encode_static_scratch(iq_format f, const void *W, iq_dtype dt, int64_t rows, int64_t cols,
                                        const float *importance, int64_t rows_per_expert, const float *grid,
                                        const uint16_t *d16, const uint8_t *choices, uint8_t *payload,
                                        float *group_errors, int32_t *status, void *stream) {
  int rc = check_common(f, W, dt, rows, cols, importance, rows_per_expert, grid);
  if (rc) return rc;
  size_t need = 0;
  iq_encode_workspace_size(f, rows, cols, &need);
  if (need > kStaticScratchBytes) return IQ_ERR_TOO_LARGE;
  void *ws = static_scratch_ptr();
  if (!ws) return IQ_ERR_CUDA;
  return iq_encode(f, W, dt, rows, cols, importance, rows_per_expert, grid, d16, choices, payload, group_errors,
                   status, ws, kStaticScratchBytes, stream);
}
