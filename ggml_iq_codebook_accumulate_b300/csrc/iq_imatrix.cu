// imatrix statistic: routed per-expert sums of squared activations and token counts
// ("Add imatrix calibration for the GGML formats and use it for fused MoE experts", What imatrix
// does: one statistic per routed expert over the tokens routed to it, rows squared 1,024 at a
// time; "MoE expert coverage in imatrix calibration", Facts: x^2 added only to the token's top-k
// experts, a per-expert token count, non-finite sums checked only for touched experts, count 0
// -> weight 1).
//
// Definition computed (bit for bit): for each chunk of rows_per_chunk tokens and each expert e the
// chunk routes tokens to, partial[e][j] starts at +0 and, over those tokens in ascending order,
// becomes fl(partial + fl(x*x)) -- the square rounded to fp32, then added with one more rounding
// (for both input types: a bf16 square is exact in fp32 unless it falls below the normal range,
// where it rounds too); then in_sum2[e][j] = fl(in_sum2[e][j] + partial[e][j]), chunk by chunk.
//
// Kernels per call:
//  route       one CTA per (chunk, sub-tile of 128 or 64 rows): builds the sub-tile's expert bitmap
//              in shared memory (a token's ids are a set) and writes the sub-tile's segment: for
//              every expert the offset and length of its run of rows, then the runs themselves
//              (32-bit byte offsets into a staged tile, ascending, each run padded to a multiple
//              of 4 with the offset of a zero row); counts per (chunk, expert) and per expert over
//              the call are added atomically;
//  accumulate  one CTA per (column tile of 512 bytes: 256 bf16 / 128 fp32 columns, part) and, when
//              there are too few to fill the GPU, per chunk as well; the parts split the experts.
//              Launched as a programmatic dependent of the route kernel, it sets up while that
//              runs.  A producer warp streams the tile's rows through a ring of up to 4
//              shared-memory stages: each stage is one 2-D TMA tensor copy of the sub-tile's rows
//              plus one bulk copy of its segment, both completing on the stage's mbarrier (all
//              waits bounded by the global timer).  Meanwhile the 12 consumer warps plan their
//              part (ranked experts, each dealt whole to the least-loaded warp); then each walks
//              its experts' rows, 4 at a time, from shared memory (a lane reads 16 bytes of a
//              row) into one register accumulator per (expert, column of its lane).  For bf16,
//              two screening warps check each landed stage for values whose squares are inexact
//              in fp32; stages without any take one mixed-precision FMA per value, the others
//              square and add separately.  With one expert (a dense statistic) 4 consumer warps
//              take 128 bytes of every row each, with no plan and no screening;
//  combine     (per-chunk mode only) adds the chunk partials to in_sum2 in chunk order.
// No atomics touch in_sum2, so the sums are the sequential definition above.
#include <cudaTypedefs.h>

#include <climits>
#include <type_traits>
#include <mutex>

#include "iq_common.cuh"

namespace iqk {

constexpr int kRowBytes = 512;      // bytes of one row of a column tile (256 bf16 / 128 fp32 columns)
constexpr int kMaxSub = 128;        // rows per stage (64 when the segments are large)
constexpr int kMaxStages = 4;       // shared-memory ring depth (fewer when stages are large)
constexpr int kSlots = 6;           // work units per consumer warp
constexpr int kMaxConsumers = 12;   // consumer warps per CTA: 3 per warp scheduler
constexpr int kPartUnits = kMaxConsumers * kSlots;  // units one CTA (part) can hold
constexpr int kMaxParts = 16;       // CTAs that share a column tile, each with its own experts
constexpr int kMinSeqCtas = 112;    // below this many (tile, part) CTAs, chunks also run in parallel
constexpr int kMaxTopK = 64;        // bounds the rows a segment holds
constexpr size_t kSmemBudget = 216 * 1024;   // stages; the kernel's static arrays take 7 KB more

template <typename T> struct Col;
template <> struct Col<__nv_bfloat16> { static constexpr int TILE = 256; };
template <> struct Col<float> { static constexpr int TILE = 128; };

__host__ __device__ inline size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

__host__ __device__ inline int align16(int n) { return (n + 15) & ~15; }

// A segment (one per chunk and sub-tile of `sub` rows): int2 (start, length) per expert (padded to
// 16 bytes), then the rows of expert 0, expert 1, ... as uint32 byte offsets (row * 512) into the
// staged tile, each run ascending and padded to a multiple of 4 entries (so a run starts on a
// 16-byte boundary) with the offset of the zero row that follows the tile.
struct SegLayout {
  int offb;   // bytes of the (start, length) table
  int bytes;  // segment bytes (multiple of 16)
};
__host__ __device__ inline SegLayout seg_layout(int E, int top_k, int sub) {
  SegLayout l;
  l.offb = align16(E * 8);
  l.bytes = l.offb + align16(4 * (sub * (top_k < E ? top_k : E) + 3 * E));
  return l;
}

// A work unit of the accumulation is one expert over the tile's columns; a consumer warp's plan
// slot holds its id, or -1 (no unit).

struct RouteWs {
  int32_t *touched;    // [E]   experts this call routed at least one token to
  int32_t *ccount;     // [nchunks][E] tokens per (chunk, expert)
  int32_t *ecount;     // [E]   tokens per expert over the call
  uint8_t *seg;        // [nchunks][nsub] segments of seg_bytes
  float *partial;      // [nchunks][E][cols] (per-chunk mode only)
  size_t zero_bytes;   // bytes from the start to clear before the call (touched, ccount, ecount)
};

struct Plan {
  int64_t nchunks, ntiles;
  int nsub, sub, nparts, nstages, stage_bytes;
  SegLayout seg;
  bool split;
};

static Plan make_plan(int64_t tokens, int64_t cols, iq_dtype dt, int E, int top_k, int64_t rpc, int sms) {
  Plan p;
  p.nchunks = (tokens + rpc - 1) / rpc;
  // stages of 128 rows, or 64 when three stages with their segments would not fit
  p.sub = kMaxSub;
  for (;;) {
    p.seg = seg_layout(E, top_k, p.sub);
    p.stage_bytes = (p.sub * kRowBytes + kRowBytes + p.seg.bytes + 127) & ~127;
    if (p.sub == 64 || 3 * (size_t)p.stage_bytes <= kSmemBudget) break;
    p.sub = 64;
  }
  p.nstages = (int)(kSmemBudget / (size_t)p.stage_bytes);
  if (p.nstages > kMaxStages) p.nstages = kMaxStages;
  if (p.nstages < 2) p.nstages = 2;
  p.nsub = (int)((rpc + p.sub - 1) / p.sub);
  const int tile = dt == IQ_BF16 ? Col<__nv_bfloat16>::TILE : Col<float>::TILE;
  p.ntiles = (cols + tile - 1) / tile;
  // parts per tile: enough that a part's experts fit its warps' slots, and as many as fill the
  // SMs (at most one per expert)
  const int need = (E + kPartUnits - 1) / kPartUnits;
  int fill = (int)(sms / p.ntiles);
  if (fill > E) fill = E;
  if (fill > kMaxParts) fill = kMaxParts;
  if (fill < 1) fill = 1;
  p.nparts = need > fill ? need : fill;
  p.split = p.nchunks > 1 && p.ntiles * p.nparts < kMinSeqCtas;
  return p;
}

static RouteWs route_ws(void *ws, const Plan &p, int E, int64_t cols) {
  uint8_t *q = (uint8_t *)ws;
  RouteWs r;
  r.touched = (int32_t *)q; q += align256((size_t)E * 4);
  r.ccount = (int32_t *)q; q += align256((size_t)p.nchunks * E * 4);
  r.ecount = (int32_t *)q; q += align256((size_t)E * 4);
  r.zero_bytes = (size_t)(q - (uint8_t *)ws);
  r.seg = q; q += align256((size_t)p.nchunks * p.nsub * p.seg.bytes);
  r.partial = p.split ? (float *)q : nullptr;
  return r;
}
static size_t route_ws_bytes(const Plan &p, int E, int64_t cols) {
  size_t n = align256((size_t)E * 4) + align256((size_t)p.nchunks * E * 4) + align256((size_t)E * 4) +
             align256((size_t)p.nchunks * p.nsub * p.seg.bytes);
  if (p.split) n += align256((size_t)p.nchunks * E * cols * 4);
  return n;
}

// ---------------------------------------------------------------------------------------------
// bar.sync on barrier `id` (1..15) for `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// The work plan of one part (the CTAs with this blockIdx.z share a column tile's experts), built by
// the consumer warps of every CTA from the counts over the whole call (the same plan for every
// chunk and tile, so each (expert, column) sum has one owner warp).  Experts are ranked by count
// (ties: lower id) and dealt to the parts in snake order of rank; a part's experts, in rank order,
// go one by one to the consumer warp with the least work so far among those with a free slot
// (ties: lower warp).  An expert's work is its rows plus a fixed cost for each stage it has rows
// in (a run starts with two dependent shared-memory loads, and is padded to whole groups of 4):
// c + 4 min(c, stages).  Cutting heavy experts into column parts was measured slower: the narrower
// loads cost more per row than the better balance gains, as a long run streams at full speed.
//   cnt: [E] scratch (the counts), rank: [E] scratch, ul: [kPartUnits] scratch, ud: the plan slots;
//   bar: a named barrier over the nthreads consumer threads (tid = their index).
__device__ void plan_part(const int32_t *__restrict__ ecount, int E, int nparts, int p, int64_t stages, int *cnt,
                          int16_t *rank, int2 *ul, int (*ud)[kSlots], int tid, int nthreads, int bar) {
  for (int e = tid; e < E; e += nthreads) cnt[e] = ecount[e];
  for (int i = tid; i < kMaxConsumers * kSlots; i += nthreads) ud[i / kSlots][i % kSlots] = -1;
  named_barrier(bar, nthreads);
  // rank by counting: experts ahead of e have a larger count, or the same count and a lower id
  for (int e = tid; e < E; e += nthreads) {
    const int c = cnt[e];
    int r = 0;
#pragma unroll 8
    for (int j = 0; j < E; j++) {
      const int cj = cnt[j];
      r += (cj > c) | ((cj == c) & (j < e));
    }
    rank[r] = (int16_t)e;
  }
  named_barrier(bar, nthreads);
  if (tid < 32) {
    const int lane = tid;
    const int nexp = (E + nparts - 1) / nparts;          // bound on the part's experts (ranks < E)
    int base = 0;
    for (int l0 = 0; l0 < nexp; l0 += 32) {              // the part's experts with rows, in rank order
      const int l = l0 + lane;
      const int r = l * nparts + ((l & 1) ? nparts - 1 - p : p);
      int e = 0, c = 0;
      if (l < nexp && r < E) { e = rank[r]; c = cnt[e]; }
      const unsigned has = __ballot_sync(0xffffffffu, c > 0);
      const int ui = base + __popc(has & ((1u << lane) - 1u));
      if (c > 0 && ui < kPartUnits) {
        const int64_t w = (int64_t)c + 4 * min((int64_t)c, stages);
        ul[ui] = make_int2(e, (int)min(w, (int64_t)0x0fffffff));
      }
      base += __popc(has);
    }
    __syncwarp();
    // deal: the (load, warp) minimum over the warps with a free slot is one warp-wide reduction of
    // load << 4 | warp (loads saturate at 2^28 - 1; a warp with a free slot always wins over one
    // without, as the all-ones key needs lane 15)
    const int nu = min(base, kPartUnits);
    uint32_t load = 0;
    int nslot = 0;
    for (int u0 = 0; u0 < nu; u0 += 32) {                // 32 units at a time, one per lane
      const int2 mine = u0 + lane < nu ? ul[u0 + lane] : make_int2(-1, 0);
      const int n = min(32, nu - u0);
#pragma unroll 4
      for (int j = 0; j < n; j++) {
        const int dx = __shfl_sync(0xffffffffu, mine.x, j), dy = __shfl_sync(0xffffffffu, mine.y, j);
        const uint32_t k = lane < kMaxConsumers && nslot < kSlots ? load << 4 | (uint32_t)lane : 0xffffffffu;
        const uint32_t w = __reduce_min_sync(0xffffffffu, k) & 15u;
        if (lane == (int)w) {
          ud[w][nslot] = dx;
          load = min(load + (uint32_t)dy, 0x0fffffffu);
          nslot++;
        }
      }
    }
  }
  named_barrier(bar, nthreads);
}

// One CTA per (sub-tile s, chunk k): rows [sub * s, sub * s + sub) of chunk k.
__global__ void __launch_bounds__(256) imatrix_route(const int32_t *__restrict__ ids, int64_t tokens, int top_k,
                                                     int E, int64_t rpc, int nsub, int sub, SegLayout sl, RouteWs ws,
                                                     unsigned long long *__restrict__ counts,
                                                     int32_t *__restrict__ status) {
  __shared__ uint32_t bm[1024][kMaxSub / 32];   // expert x row bitmap of the sub-tile
  __shared__ int cnt[1024 + 1], off[1024 + 1];
  __shared__ int wtot[8];                        // the scan's warp totals (256 threads)
  // the accumulate kernel may be scheduled now: it waits for this grid's completion itself
  asm volatile("griddepcontrol.launch_dependents;");
  const int words = sub / 32;
  const int s = blockIdx.x;
  const int64_t k = blockIdx.y;
  const int64_t r0 = k * rpc + (int64_t)s * sub;
  const int64_t rend = min(tokens, (k + 1) * rpc);
  const int rows = (int)max((int64_t)0, min((int64_t)sub, rend - r0));
  for (int i = threadIdx.x; i < E * words; i += blockDim.x) bm[i / words][i % words] = 0u;
  __syncthreads();
  // a unit is one slot of 32 consecutive rows; the lanes holding the same expert set their bits
  // with one atomic (the rows of a 32-row group are one bitmap word).  A bit that is already set
  // is the same (row, expert) from another slot: a repeated id, which the bitmap counts once.  A
  // warp loads the ids of up to 8 of its units before it sets their bits.
  int st = 0;
  const int lane = threadIdx.x & 31, groups = (rows + 31) / 32, nunits = groups * top_k;
  const int nw = blockDim.x >> 5;
  for (int u0 = threadIdx.x >> 5; u0 < nunits; u0 += 8 * nw) {
    int ev[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const int idx = u0 + j * nw, g = idx % groups, a = idx / groups, r = g * 32 + lane;
      ev[j] = idx < nunits && r < rows ? ids[(r0 + r) * top_k + a] : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const int idx = u0 + j * nw;
      if (idx >= nunits) break;  // the same in every lane
      const int g = idx % groups;
      const bool in = g * 32 + lane < rows;
      int e = ev[j];
      if (in && (e < 0 || e >= E)) st |= IQ_STATUS_BAD_EXPERT_ID;
      if (!in || e < 0 || e >= E) e = -1;
      const unsigned same = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(same) - 1 && (atomicOr(&bm[e][g], same) & same))
        st |= IQ_STATUS_DUP_EXPERT_ID;
    }
  }
  if (st && status) atomicOr(status, st);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < words; w++) c += __popc(bm[e][w]);
    cnt[e] = c;
  }
  __syncthreads();
  {  // exclusive scan of the padded run lengths over experts: 4 consecutive experts a thread
     // (256 x 4 >= 1024 >= E), a warp scan of the threads' sums, then the warps' totals
    const int e0 = threadIdx.x * 4, warp = threadIdx.x >> 5;
    int v[4], tsum = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
      v[j] = e0 + j < E ? (cnt[e0 + j] + 3) & ~3 : 0;
      tsum += v[j];
    }
    int incl = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    int p = incl - tsum;
    for (int w = 0; w < warp; w++) p += wtot[w];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      if (e0 + j < E) off[e0 + j] = p;
      p += v[j];
    }
  }
  __syncthreads();
  uint8_t *seg = ws.seg + ((size_t)k * nsub + s) * sl.bytes;
  int2 *sse = reinterpret_cast<int2 *>(seg);
  uint32_t *srow = reinterpret_cast<uint32_t *>(seg + sl.offb);
  const uint32_t zero_off = (uint32_t)(sub * kRowBytes);
  // runs: one thread per (expert, bitmap word) writes the word's rows at the word's position in
  // the expert's run; the last word's thread pads the run to a multiple of 4
  for (int i = threadIdx.x; i < E * words; i += blockDim.x) {
    const int e = i / words, w = i % words;
    int p = off[e];
    for (int v = 0; v < w; v++) p += __popc(bm[e][v]);
    uint32_t word = bm[e][w];
    while (word) {
      const int bit = __ffs(word) - 1;
      word &= word - 1;
      srow[p++] = (uint32_t)((w * 32 + bit) * kRowBytes);
    }
    if (w == words - 1) {
      sse[e] = make_int2(off[e], cnt[e]);
      while (p & 3) srow[p++] = zero_off;
    }
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = cnt[e];
    if (c) {
      atomicAdd(&ws.ccount[(size_t)k * E + e], c);
      atomicAdd(&ws.ecount[e], c);
      atomicAdd(&counts[e], (unsigned long long)c);
      ws.touched[e] = 1;
    }
  }
}

// ---------------------------------------------------------------------------------------------
struct AccArgs {
  int64_t tokens, cols, rpc, nchunks;
  int E, nsub, sub, stage_bytes, nstages;
  SegLayout sl;
  RouteWs ws;
  float *in_sum2;
  int32_t *status;
  uint64_t neg0;   // -0.0f in both 32-bit halves
};

// Shared-memory loads through 32-bit shared-window addresses (explicitly the shared state space;
// volatile so they stay after the stage's mbarrier wait).
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ int2 lds_i2(uint32_t a) {
  int2 v;
  asm volatile("ld.shared.v2.s32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

// acc += x^2 for the lane's values of one row: the square rounded to fp32, then added with one more
// rounding, two columns per instruction (packed fp32x2, round to nearest, no flush).  The square is
// formed as fma(x, x, z) with z = -0 in both halves (x*x + -0 = x*x, also for +0, so it is x*x
// rounded once).  z is a kernel argument: with a literal -0 the compiler turns the fma into a
// multiply and fuses that with the add, which rounds once and differs where the square is inexact
// (fp32 inputs; bf16 inputs whose squares fall below the normal range).  A bf16 value widens to
// fp32 exactly by moving its bits to the upper half.
__device__ __forceinline__ void sq_add2(float &a0, float &a1, float x0, float x1, uint64_t z) {
  unsigned long long acc, x;
  asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
  asm("fma.rn.f32x2 %0, %0, %0, %1;" : "+l"(x) : "l"(z));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc) : "l"(x));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc));
}
// bf16, EX: the square rounded, then added (packed as above).  bf16, !EX: one mixed-precision FMA
// per value, acc = fl(acc + x*x) with one rounding -- the same value whenever x*x is exact in fp32,
// which holds for every bf16 x with |x| >= 2^-67 or x = 0 (8 significant bits, so x*x has at
// most 16 and stays above the subnormal step 2^-149); stages holding a value below that take EX.
template <bool EX> __device__ __forceinline__ void sq_add_bf16x2(float &a0, float &a1, uint32_t u, uint64_t z) {
  if (EX) {
    sq_add2(a0, a1, __uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u), z);
  } else {
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n fma.rn.f32.bf16 %0, l, l, %0;\n fma.rn.f32.bf16 %1, h, h, %1;\n}\n"
        : "+f"(a0), "+f"(a1) : "r"(u));
  }
}
// One row of a unit: the lane's 16 bytes of the staged tile (8 bf16 or 4 fp32 values).
template <typename T, bool EX> struct AccRow;
template <bool EX> struct AccRow<__nv_bfloat16, EX> {
  static __device__ __forceinline__ void run(float *acc, const uint4 &v, uint64_t z) {
    sq_add_bf16x2<EX>(acc[0], acc[1], v.x, z); sq_add_bf16x2<EX>(acc[2], acc[3], v.y, z);
    sq_add_bf16x2<EX>(acc[4], acc[5], v.z, z); sq_add_bf16x2<EX>(acc[6], acc[7], v.w, z);
  }
};
template <bool EX> struct AccRow<float, EX> {
  static __device__ __forceinline__ void run(float *acc, const uint4 &v, uint64_t z) {
    sq_add2(acc[0], acc[1], __uint_as_float(v.x), __uint_as_float(v.y), z);
    sq_add2(acc[2], acc[3], __uint_as_float(v.z), __uint_as_float(v.w), z);
  }
};
// The n >= 1 rows of one unit in this stage, in ascending order.  srow: shared address of the unit's
// first row offset (16-byte aligned); base: the lane's first byte in the staged tile.  The run is
// padded with the zero row's offset to whole groups of 4, and a zero row adds exactly nothing
// (fl(acc + 0) = acc for acc >= +0), so every group is whole; groups are software pipelined
// (offsets two groups ahead of the additions, rows one group ahead).
template <typename T, bool EX>
__device__ __forceinline__ void run_unit(float *acc, uint32_t srow, int n, uint32_t base, uint64_t z) {
  using A = AccRow<T, EX>;
  const int n4 = (n + 3) & ~3;
  const uint4 o = lds_v4(srow);
  uint4 on = lds_v4(srow + 4 * min(4, n4 - 4));
  uint4 r0 = lds_v4(base + o.x), r1 = lds_v4(base + o.y), r2 = lds_v4(base + o.z), r3 = lds_v4(base + o.w);
#pragma unroll 1
  for (int j = 4; j < n4; j += 4) {
    const uint4 onn = lds_v4(srow + 4 * min(j + 4, n4 - 4));
    const uint4 n0 = lds_v4(base + on.x), n1 = lds_v4(base + on.y), n2 = lds_v4(base + on.z), n3 = lds_v4(base + on.w);
    A::run(acc, r0, z); A::run(acc, r1, z); A::run(acc, r2, z); A::run(acc, r3, z);
    r0 = n0; r1 = n1; r2 = n2; r3 = n3;
    on = onn;
  }
  A::run(acc, r0, z); A::run(acc, r1, z); A::run(acc, r2, z); A::run(acc, r3, z);
}

// One expert over the whole tile (a dense statistic): a warp takes 128 bytes of each row, a lane 4
// (2 bf16 or 1 fp32 value), squared then added with two roundings; the run is padded to whole
// groups of 4 as above.
template <typename T>
__device__ __forceinline__ void run_dense(float *acc, uint32_t srow, int n, uint32_t base, uint64_t z) {
  auto add = [&](uint32_t u) {
    if (std::is_same<T, __nv_bfloat16>::value) sq_add_bf16x2<true>(acc[0], acc[1], u, z);
    else { const float x = __uint_as_float(u); acc[0] = __fadd_rn(acc[0], __fmul_rn(x, x)); }
  };
  const int n4 = (n + 3) & ~3;
  uint4 o = lds_v4(srow);
#pragma unroll 1
  for (int j = 0; j < n4; j += 4) {
    const uint4 on = lds_v4(srow + 4 * min(j + 4, n4 - 4));
    const uint32_t r0 = lds_u32(base + o.x), r1 = lds_u32(base + o.y), r2 = lds_u32(base + o.z), r3 = lds_u32(base + o.w);
    add(r0); add(r1); add(r2); add(r3);
    o = on;
  }
}

// The lane's NV (8 for bf16, 4 for fp32) current sums at src (16-byte aligned).
template <int NV> __device__ __forceinline__ void load_unit(const float *src, float *v) {
#pragma unroll
  for (int i = 0; i < NV; i += 4) {
    const float4 t = *reinterpret_cast<const float4 *>(src + i);
    v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
  }
}
// dst = old + acc (add: in_sum2 += the lane's sums, one rounding each), or dst = acc (the chunk
// partial, for the ordered combine).  Returns whether every stored value is finite.
template <int NV> __device__ __forceinline__ bool store_unit(float *dst, const float *acc, const float *old, bool add) {
  bool fin = true;
#pragma unroll
  for (int i = 0; i < NV; i += 4) {
    float o[4];
#pragma unroll
    for (int c = 0; c < 4; c++) {
      o[c] = add ? __fadd_rn(old[i + c], acc[i + c]) : acc[i + c];
      fin &= isfinite(o[c]);
    }
    *reinterpret_cast<float4 *>(dst + i) = make_float4(o[0], o[1], o[2], o[3]);
  }
  return fin;
}

// One stage for one consumer warp: every unit of the warp (udw: its plan slots) adds the rows the
// stage routes to its expert.  hit gathers the slots that saw rows.
template <typename T, bool EX>
__device__ __forceinline__ void stage_units(float (*acc)[8], const int *udw, uint32_t stage, uint32_t sse,
                                            uint32_t srow, int lane, uint32_t &hit, uint64_t z) {
#pragma unroll
  for (int s = 0; s < kSlots; s++) {
    const int d = udw[s];
    if (d < 0) continue;
    const int2 se = lds_i2(sse + 8 * d);
    if (se.y == 0) continue;
    hit |= 1u << s;
    run_unit<T, EX>(acc[s], srow + 4 * se.x, se.y, stage + lane * 16, z);
  }
}

constexpr int kScreenWarps = 2;

// Whether a landed bf16 stage holds a value whose square is inexact in fp32 (flagged
// conservatively: 0 < |x| < 2^-63, exponent field below 64).  Screening warp sw of kScreenWarps
// reads rows sw, sw + kScreenWarps, ... (lane: 16 bytes of each): first the least magnitude per
// lane and half (one bf16x2 minimum of magnitudes per word; NaN operands are passed over), then,
// only if that is below 2^-63 or zero, the exact test.
__device__ __forceinline__ bool stage_has_tiny(uint32_t tile, int rows, int sw, int lane) {
  uint32_t m = 0x7f7f7f7fu;   // the largest finite bf16 in both halves
#pragma unroll 4
  for (int r = sw; r < rows; r += kScreenWarps) {
    const uint4 v = lds_v4(tile + (uint32_t)r * kRowBytes + lane * 16);
    asm("min.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v.x));
    asm("min.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v.y));
    asm("min.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v.z));
    asm("min.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v.w));
  }
  const bool low = (m & 0x7fffu) < 0x2000u || ((m >> 16) & 0x7fffu) < 0x2000u;
  if (!__any_sync(0xffffffffu, low)) return false;
  auto tiny = [](uint32_t h) { return ((h & 0x7fffu) - 1u) < 0x1fffu; };
  bool t = false;
#pragma unroll 4
  for (int r = sw; r < rows; r += kScreenWarps) {
    const uint4 v = lds_v4(tile + (uint32_t)r * kRowBytes + lane * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) t |= tiny(w[i] & 0xffffu) | tiny(w[i] >> 16);
  }
  return __any_sync(0xffffffffu, t);
}

// 13 warps (fp32) or 15 (bf16: two screening warps): at most 128 registers a thread, as each warp
// scheduler's quarter of the register file (16,384) must hold its warps (4 x 32 x 128).  A dense
// statistic (one expert) runs 4 consumer warps, one per 128 bytes of the tile, and the producer.
constexpr int kDenseWarps = 4;
template <typename T, bool DENSE> constexpr int acc_warps() {
  return DENSE ? kDenseWarps + 1 : kMaxConsumers + 1 + (std::is_same<T, __nv_bfloat16>::value ? kScreenWarps : 0);
}
template <typename T, bool DENSE>
__global__ void __launch_bounds__(32 * 16, 1) imatrix_accumulate_kernel(
    const __grid_constant__ CUtensorMap tmap, AccArgs a) {
  constexpr int TILE = Col<T>::TILE;
  constexpr int ESZ = (int)sizeof(T);
  const uint32_t kTileBytes = (uint32_t)(a.sub * kRowBytes);
  const uint32_t kSegOff = kTileBytes + kRowBytes;       // after the tile and its zero row
  const uint32_t kStageBytes = (uint32_t)a.stage_bytes;  // tile + zero row + segment, multiple of 128
  const int NS = a.nstages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // stage buffers start on a 128-byte boundary (one spare 128 bytes is allocated for this)
  uint8_t *smem = smem_raw + ((128 - (smem_u32(smem_raw) & 127)) & 127);
  const uint32_t smem_s = smem_u32(smem);
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages], chk_bar[kMaxStages];
  __shared__ int abort_flag, tiny_flag[kMaxStages][kScreenWarps];
  constexpr bool kScan = std::is_same<T, __nv_bfloat16>::value && !DENSE;   // bf16 stages are screened
  __shared__ int ud[kMaxConsumers][kSlots];  // the consumer warps' work units (the plan)
  __shared__ int16_t rank[1024];              // plan scratch: experts by rank
  __shared__ int cnts[1024];                  // plan scratch: the counts over the call
  __shared__ int2 ul[kPartUnits];             // plan scratch: the part's units

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = DENSE ? kDenseWarps : kMaxConsumers;
  const int64_t col0 = (int64_t)blockIdx.x * TILE;
  const bool split = a.ws.partial != nullptr;
  const int64_t kbeg = split ? blockIdx.y : 0, kend = split ? blockIdx.y + 1 : a.nchunks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; s++) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], NW); mbar_init(&chk_bar[s], kScreenWarps); }
    abort_flag = 0;
    mbar_fence_init();
  }
  // the row after the tile in every stage is a zero row: a group of row offsets is padded with it
  for (int i = threadIdx.x; i < NS * kRowBytes / 4; i += blockDim.x)
    reinterpret_cast<uint32_t *>(smem + (size_t)(i / (kRowBytes / 4)) * kStageBytes + kTileBytes)[i % (kRowBytes / 4)] = 0u;
  // the route kernel (segments, counts) is complete and visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  // the consumers plan the part while the producer starts the first stages
  if (!DENSE && warp < NW)
    plan_part(a.ws.ecount, a.E, gridDim.z, blockIdx.z, a.nchunks * a.nsub, cnts, rank, ul, ud, threadIdx.x, NW * 32, 1);

  if (warp == NW) {
    // ---- producer: lane 0 issues the tile's row stages in consumption order --------------
    if (lane == 0) {
      int64_t q = 0;
      bool ok = true;
      for (int64_t k = kbeg; k < kend && ok; k++) {
        const int64_t rows = min(a.rpc, a.tokens - k * a.rpc);
        const int nsub = (int)((rows + a.sub - 1) / a.sub);
        for (int sub = 0; sub < nsub && ok; sub++, q++) {
          const int st = (int)(q % NS);
          if (q >= NS) ok = mbar_wait_bounded(&empty_bar[st], (uint32_t)((q / NS - 1) & 1));
          if (!ok || *(volatile int *)&abort_flag) { ok = false; break; }
          uint8_t *dst = smem + (size_t)st * kStageBytes;
          mbar_expect_tx(&full_bar[st], kTileBytes + (uint32_t)a.sl.bytes);
          tma_load_2d(dst, &tmap, (int)col0, (int)(k * a.rpc + (int64_t)sub * a.sub), &full_bar[st]);
          bulk_copy_g2s(dst + kSegOff, a.ws.seg + ((size_t)k * a.nsub + sub) * a.sl.bytes, (uint32_t)a.sl.bytes,
                        &full_bar[st]);
        }
      }
      if (!ok) {
        atomicExch(&abort_flag, 1);
        if (a.status) atomicOr(a.status, IQ_STATUS_TIMEOUT);
      }
      // every issued copy must land before the CTA's shared memory is released
      for (int64_t u = q - NS < 0 ? 0 : q - NS; u < q; u++)
        mbar_wait_bounded(&full_bar[u % NS], (uint32_t)((u / NS) & 1));
    }
  } else if (warp > NW) {
    // ---- bf16 screening warps: each stage as it lands, every kScreenWarps-th row each ------------
    const int sw = warp - NW - 1;
    int64_t q = 0;
    bool ok = true;
    for (int64_t k = kbeg; k < kend && ok; k++) {
      const int64_t rows = min(a.rpc, a.tokens - k * a.rpc);
      const int nsub = (int)((rows + a.sub - 1) / a.sub);
      for (int sub = 0; sub < nsub && ok; sub++, q++) {
        const int st = (int)(q % NS);
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full_bar[st], (uint32_t)((q / NS) & 1)));
        if (!ok || *(volatile int *)&abort_flag) { ok = false; break; }
        const bool t = stage_has_tiny(smem_s + (uint32_t)st * kStageBytes, a.sub, sw, lane);
        if (lane == 0) {
          *(volatile int *)&tiny_flag[st][sw] = t ? 1 : 0;
          mbar_arrive(&chk_bar[st]);
        }
      }
    }
    if (!ok && lane == 0) {
      atomicExch(&abort_flag, 1);
      if (a.status) atomicOr(a.status, IQ_STATUS_TIMEOUT);
    }
  } else if (DENSE) {
    // ---- dense consumers: warp w takes bytes [128 w, 128 w + 128) of every row --------------------
    constexpr int NV = 4 / ESZ;
    const uint32_t lb = (uint32_t)(warp * 128 + lane * 4);
    int64_t q = 0;
    bool ok = true, fin = true;
    for (int64_t k = kbeg; k < kend && ok; k++) {
      const int64_t rows = min(a.rpc, a.tokens - k * a.rpc);
      const int nsub = (int)((rows + a.sub - 1) / a.sub);
      float acc[2] = {0.0f, 0.0f};
      bool hit = false;
      for (int sub = 0; sub < nsub; sub++, q++) {
        const int st = (int)(q % NS);
        if (!mbar_wait_bounded(&full_bar[st], (uint32_t)((q / NS) & 1)) || *(volatile int *)&abort_flag) {
          ok = false;
          break;
        }
        const uint32_t stage = smem_s + (uint32_t)st * kStageBytes;
        const uint32_t sse = stage + kSegOff, srow = sse + (uint32_t)a.sl.offb;
        const int2 se = lds_i2(sse);
        if (se.y > 0) {
          hit = true;
          run_dense<T>(acc, srow + 4 * se.x, se.y, stage + lb, a.neg0);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[st]);
      }
      if (!ok) break;
      const int64_t c = col0 + lb / ESZ;
      if (hit && c < a.cols) {
        float *p = split ? a.ws.partial + (size_t)k * a.cols + c : a.in_sum2 + c;
#pragma unroll
        for (int i = 0; i < NV; i++) {
          const float v = split ? acc[i] : __fadd_rn(p[i], acc[i]);
          p[i] = v;
          fin &= isfinite(v);
        }
      }
    }
    if (!ok && lane == 0) {
      atomicExch(&abort_flag, 1);
      if (a.status) atomicOr(a.status, IQ_STATUS_TIMEOUT);
    }
    if (!split && a.status && __any_sync(0xffffffffu, !fin) && lane == 0) atomicOr(a.status, IQ_STATUS_NONFINITE_SUM2);
  } else {
    // ---- consumers: each warp walks its units (plan) over every stage --------------------------
    int64_t q = 0;
    bool ok = true, fin = true;
    for (int64_t k = kbeg; k < kend && ok; k++) {
      const int64_t rows = min(a.rpc, a.tokens - k * a.rpc);
      const int nsub = (int)((rows + a.sub - 1) / a.sub);
      float acc[kSlots][8];
      uint32_t hit = 0;   // slots whose expert has rows in this chunk
#pragma unroll
      for (int s = 0; s < kSlots; s++)
#pragma unroll
        for (int c = 0; c < 8; c++) acc[s][c] = 0.0f;
      for (int sub = 0; sub < nsub; sub++, q++) {
        const int st = (int)(q % NS);
        const uint32_t par = (uint32_t)((q / NS) & 1);
        if ((kScan && !mbar_wait_bounded(&chk_bar[st], par)) || !mbar_wait_bounded(&full_bar[st], par) ||
            *(volatile int *)&abort_flag) {
          ok = false;
          break;
        }
        const uint32_t stage = smem_s + (uint32_t)st * kStageBytes;
        const uint32_t sse = stage + kSegOff, srow = sse + (uint32_t)a.sl.offb;
        if (!kScan || (*(volatile int *)&tiny_flag[st][0] | *(volatile int *)&tiny_flag[st][1]))
          stage_units<T, true>(acc, ud[warp], stage, sse, srow, lane, hit, a.neg0);
        else
          stage_units<T, false>(acc, ud[warp], stage, sse, srow, lane, hit, a.neg0);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[st]);
      }
      if (!ok) break;
      // chunk done: add the partials to in_sum2 (or store them for the ordered combine), for the
      // experts the chunk routed rows to (every part of an expert sees the same rows).  The
      // current sums of half the slots at a time are loaded first, so their latencies overlap.
      auto unit_dst = [&](int s) -> float * {
        const int d = ud[warp][s];
        if (d < 0 || !((hit >> s) & 1u)) return nullptr;
        const int e = d;
        const int64_t c = col0 + lane * (16 / ESZ);
        if (c >= a.cols) return nullptr;
        return split ? a.ws.partial + ((size_t)k * a.E + e) * a.cols + c : a.in_sum2 + (size_t)e * a.cols + c;
      };
      constexpr int kHalf = (kSlots + 1) / 2;
#pragma unroll
      for (int h = 0; h < kSlots; h += kHalf) {
        float old[kHalf][8];
#pragma unroll
        for (int s = h; s < h + kHalf && s < kSlots; s++) {
          const float *p = unit_dst(s);
          if (p && !split) load_unit<16 / ESZ>(p, old[s - h]);
        }
#pragma unroll
        for (int s = h; s < h + kHalf && s < kSlots; s++) {
          float *p = unit_dst(s);
          if (p) fin &= store_unit<16 / ESZ>(p, acc[s], old[s - h], !split);
        }
      }
    }
    if (!ok && lane == 0) {
      atomicExch(&abort_flag, 1);
      if (a.status) atomicOr(a.status, IQ_STATUS_TIMEOUT);
    }
    // non-finite sums of the touched experts (sequential mode: every touched expert's columns of
    // this tile were stored by their unit's lanes at least once, the last time with the final
    // sum; the combine kernel checks in per-chunk mode)
    if (!split && a.status && __any_sync(0xffffffffu, !fin) && lane == 0) atomicOr(a.status, IQ_STATUS_NONFINITE_SUM2);
  }
  __syncthreads();
}

// per-chunk mode: in_sum2 += partial[k] for k = 0, 1, ... (experts the chunk routed tokens to)
__global__ void __launch_bounds__(256) imatrix_combine(int64_t cols, int E, int64_t nchunks, RouteWs ws,
                                                       float *__restrict__ in_sum2, int32_t *__restrict__ status) {
  const int64_t n = (int64_t)E * cols;
  int bad = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / cols);
    if (!ws.touched[e]) continue;
    float v = in_sum2[i];
    for (int64_t k = 0; k < nchunks; k++)
      if (ws.ccount[(size_t)k * E + e]) v = __fadd_rn(v, ws.partial[(size_t)k * E * cols + i]);
    in_sum2[i] = v;
    bad |= !isfinite(v);
  }
  if (status && __any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, IQ_STATUS_NONFINITE_SUM2);
}

// ---------------------------------------------------------------------------------------------
// Host: 2-D tensor map of x ([tokens, cols], row-major) with a box of 512 bytes x `sub` rows.
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}

static bool make_tmap(CUtensorMap *m, const void *x, iq_dtype dt, int64_t tokens, int64_t cols, int sub) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int esz = dt == IQ_BF16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)tokens};
  cuuint64_t strides[1] = {(cuuint64_t)cols * esz};
  cuuint32_t box[2] = {(cuuint32_t)(kRowBytes / esz), (cuuint32_t)sub};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt == IQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
            const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, bool DENSE>
static int launch_accumulate(const CUtensorMap &tm, const AccArgs &a, const Plan &p, cudaStream_t st) {
  const size_t smem = (size_t)a.nstages * a.stage_bytes + 128;
  auto kern = imatrix_accumulate_kernel<T, DENSE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return IQ_ERR_CUDA;
  // programmatic dependent launch: the CTAs start (barriers, zero rows) while the route kernel
  // runs and wait for its completion before reading what it wrote
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.ntiles, p.split ? (unsigned)p.nchunks : 1u, (unsigned)p.nparts);
  cfg.blockDim = dim3(32 * acc_warps<T, DENSE>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tm, a) != cudaSuccess) return IQ_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? IQ_OK : IQ_ERR_CUDA;
}

// The plan is laid out for this many SMs (the B300's count), so that the workspace size does not
// depend on the device the call runs on; another count changes only how well the CTAs fill it.
constexpr int kPlanSms = 148;

}  // namespace iqk

using namespace iqk;

extern "C" int iq_imatrix_workspace_size(int64_t tokens, int64_t cols, iq_dtype dt, int num_experts, int top_k,
                                         int64_t rows_per_chunk, size_t *bytes) {
  if (!bytes || tokens < 0 || cols <= 0 || (dt != IQ_F32 && dt != IQ_BF16) || num_experts <= 0 ||
      num_experts > 1024 || top_k < 1 || top_k > kMaxTopK || rows_per_chunk <= 0 || rows_per_chunk > 4096)
    return IQ_ERR_ARG;
  const Plan p = make_plan(tokens, cols, dt, num_experts, top_k, rows_per_chunk, kPlanSms);
  *bytes = route_ws_bytes(p, num_experts, cols);
  return IQ_OK;
}

extern "C" int iq_imatrix_accumulate(const void *x, iq_dtype dt, int64_t tokens, int64_t cols,
                                     const int32_t *expert_ids, int top_k, int num_experts, int64_t rows_per_chunk,
                                     float *in_sum2, int64_t *counts, int32_t *status, void *workspace,
                                     size_t workspace_bytes, void *stream) {
  if (dt != IQ_F32 && dt != IQ_BF16) return IQ_ERR_ARG;
  if (tokens < 0 || tokens > INT32_MAX || cols <= 0 || cols % 64 || top_k < 1 || top_k > kMaxTopK ||
      num_experts < top_k ||
      num_experts > 1024 || rows_per_chunk < 1 || rows_per_chunk > 4096 ||
      (tokens + rows_per_chunk - 1) / rows_per_chunk > 65535)
    return IQ_ERR_ARG;
  if (!in_sum2 || !counts || (tokens > 0 && (!x || !expert_ids))) return IQ_ERR_ARG;
  if (((uintptr_t)x & 15) || ((uintptr_t)in_sum2 & 15) || ((uintptr_t)counts & 7) || ((uintptr_t)expert_ids & 3))
    return IQ_ERR_ARG;
  size_t need = 0;
  iq_imatrix_workspace_size(tokens, cols, dt, num_experts, top_k, rows_per_chunk, &need);
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255)) return IQ_ERR_WORKSPACE;
  if (tokens == 0) return IQ_OK;
  const Plan p = make_plan(tokens, cols, dt, num_experts, top_k, rows_per_chunk, kPlanSms);
  CUtensorMap tm;
  if (!make_tmap(&tm, x, dt, tokens, cols, p.sub)) return IQ_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  RouteWs ws = route_ws(workspace, p, num_experts, cols);
  if (cudaMemsetAsync(workspace, 0, ws.zero_bytes, st) != cudaSuccess) return IQ_ERR_CUDA;
  imatrix_route<<<dim3((unsigned)p.nsub, (unsigned)p.nchunks), 256, 0, st>>>(
      expert_ids, tokens, top_k, num_experts, rows_per_chunk, p.nsub, p.sub, p.seg, ws, (unsigned long long *)counts,
      status);
  if (cudaPeekAtLastError() != cudaSuccess) return IQ_ERR_CUDA;
  AccArgs a;
  a.tokens = tokens; a.cols = cols; a.rpc = rows_per_chunk; a.nchunks = p.nchunks;
  a.E = num_experts; a.nsub = p.nsub; a.sub = p.sub; a.sl = p.seg;
  a.stage_bytes = p.stage_bytes;
  a.nstages = p.nstages;
  a.ws = ws; a.in_sum2 = in_sum2; a.status = status;
  a.neg0 = 0x8000000080000000ull;
  const bool dense = num_experts == 1;
  const int rc = dt == IQ_BF16 ? (dense ? launch_accumulate<__nv_bfloat16, true>(tm, a, p, st)
                                        : launch_accumulate<__nv_bfloat16, false>(tm, a, p, st))
                               : (dense ? launch_accumulate<float, true>(tm, a, p, st)
                                        : launch_accumulate<float, false>(tm, a, p, st));
  if (rc != IQ_OK) return rc;
  if (p.split) {
    const int64_t n = (int64_t)num_experts * cols;
    const int64_t blocks = (n + 255) / 256;
    imatrix_combine<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(cols, num_experts, p.nchunks, ws,
                                                                              in_sum2, status);
    if (cudaPeekAtLastError() != cudaSuccess) return IQ_ERR_CUDA;
  }
  return IQ_OK;
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

// ---------------------------------------------------------------------------------------------
// Merging, neutral entries and coverage ("MoE expert coverage in imatrix calibration", Facts: the
// GGUF imatrix format stores in_sum2 and counts per tensor so that files can be merged; the legacy
// writer stores a zero-count expert as value 1 with count 1, a neutral entry, matching the weight
// 1 the reader gives it; saving logs the share of experts with data ("partial data (xx.xx%)") and
// "no data" when no expert has any).
namespace iqk {
// in_sum2 += src (one rounding per value); counts += src counts
__global__ void imatrix_merge_kernel(float *__restrict__ s2, int64_t *__restrict__ counts,
                                     const float *__restrict__ src, const int64_t *__restrict__ src_counts, int E,
                                     int64_t cols, int32_t *__restrict__ status) {
  const int64_t n = (int64_t)E * cols;
  int bad = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = __fadd_rn(s2[i], src[i]);
    s2[i] = v;
    bad |= !isfinite(v);
    if (i < E) counts[i] += src_counts[i];
  }
  if (status && __any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, IQ_STATUS_NONFINITE_SUM2);
}

// zero-count experts: every channel's sum becomes 1 (the count is set by a second launch, after
// every channel has read it)
__global__ void imatrix_neutral_sums_kernel(float *__restrict__ s2, const int64_t *__restrict__ counts, int E,
                                            int64_t cols) {
  const int64_t n = (int64_t)E * cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    if (counts[i / cols] == 0) s2[i] = 1.0f;
}
__global__ void imatrix_neutral_counts_kernel(int64_t *__restrict__ counts, int E) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x)
    if (counts[e] == 0) counts[e] = 1;
}

// out[0] experts with at least one token, out[1] tokens over all experts, out[2] least and out[3]
// largest count (one CTA)
__global__ void __launch_bounds__(1024) imatrix_coverage_kernel(const int64_t *__restrict__ counts, int E,
                                                                int64_t *__restrict__ out) {
  __shared__ long long r_touched[32], r_total[32], r_min[32], r_max[32];
  long long touched = 0, total = 0, mn = LLONG_MAX, mx = LLONG_MIN;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const long long c = counts[e];
    touched += c > 0;
    total += c;
    mn = c < mn ? c : mn;
    mx = c > mx ? c : mx;
  }
  for (int off = 16; off >= 1; off >>= 1) {
    touched += __shfl_xor_sync(0xffffffffu, touched, off);
    total += __shfl_xor_sync(0xffffffffu, total, off);
    const long long om = __shfl_xor_sync(0xffffffffu, mn, off), ox = __shfl_xor_sync(0xffffffffu, mx, off);
    mn = om < mn ? om : mn;
    mx = ox > mx ? ox : mx;
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { r_touched[w] = touched; r_total[w] = total; r_min[w] = mn; r_max[w] = mx; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < (int)(blockDim.x >> 5); k++) {
      touched += r_touched[k];
      total += r_total[k];
      mn = r_min[k] < mn ? r_min[k] : mn;
      mx = r_max[k] > mx ? r_max[k] : mx;
    }
    out[0] = touched;
    out[1] = total;
    out[2] = mn;
    out[3] = mx;
  }
}
}  // namespace iqk

extern "C" int iq_imatrix_merge(float *in_sum2, int64_t *counts, const float *src_in_sum2, const int64_t *src_counts,
                                int num_experts, int64_t cols, int32_t *status, void *stream) {
  if (num_experts <= 0 || cols <= 0 || !in_sum2 || !counts || !src_in_sum2 || !src_counts) return IQ_ERR_ARG;
  if (src_in_sum2 == in_sum2 || src_counts == counts) return IQ_ERR_ARG;
  const int64_t n = (int64_t)num_experts * cols;
  const int64_t blocks = (n + 255) / 256;
  iqk::imatrix_merge_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, (cudaStream_t)stream>>>(
      in_sum2, counts, src_in_sum2, src_counts, num_experts, cols, status);
  return cudaPeekAtLastError() == cudaSuccess ? IQ_OK : IQ_ERR_CUDA;
}

extern "C" int iq_imatrix_neutral_entries(float *in_sum2, int64_t *counts, int num_experts, int64_t cols,
                                          void *stream) {
  if (num_experts <= 0 || cols <= 0 || !in_sum2 || !counts) return IQ_ERR_ARG;
  const int64_t n = (int64_t)num_experts * cols;
  const int64_t blocks = (n + 255) / 256;
  cudaStream_t st = (cudaStream_t)stream;
  iqk::imatrix_neutral_sums_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(in_sum2, counts,
                                                                                          num_experts, cols);
  iqk::imatrix_neutral_counts_kernel<<<(num_experts + 255) / 256, 256, 0, st>>>(counts, num_experts);
  return cudaPeekAtLastError() == cudaSuccess ? IQ_OK : IQ_ERR_CUDA;
}

extern "C" int iq_imatrix_coverage(const int64_t *counts, int num_experts, int64_t *out, void *stream) {
  if (num_experts <= 0 || !counts || !out) return IQ_ERR_ARG;
  iqk::imatrix_coverage_kernel<<<1, 1024, 0, (cudaStream_t)stream>>>(counts, num_experts, out);
  return cudaPeekAtLastError() == cudaSuccess ? IQ_OK : IQ_ERR_CUDA;
}
