// markov_propose.cu -- the whole Markov proposal of bf16 weights in one persistent launch
// ("[DeepSeek-6] DSpark", section 4 "Markov Head": for k = 1..gamma, p_k = softmax(U_k +
// W1[x_{k-1}] W2) and x_k is drawn from p_k, so the gamma positions are serial; section 3 for
// the softmax and sampling).
//
// Why one launch. Per position, the bias GEMM on tcgen05 streams the U rows (the HBM-bound
// part), but every row then needs its token before the next position can start: the select
// (max, normaliser, crossing segment, rebuild), the gather of the drawn tokens' W1 rows into
// tensor memory and the launch gaps are serial work on a nearly idle GPU. Here the requests are
// split into groups of up to 128 rows and the positions of different groups are pipelined:
// while one group's rows are selected and their next A operand is gathered, the tensor cores
// and the copy engines stream the next group. Requests are independent, so this changes only
// the order of the work, not its arithmetic.
//
// Sweep s (s = 0 .. gamma*G - 1) is position k = s / G + 1 of group g = s % G: one pass over
// all 128-column W2 tiles against the group's 128-row block.
// CTAs (one per SM, all resident; a launch that cannot hold them all times out, it cannot hang):
//   streaming CTAs (the SMs left after the select CTAs and, with a target, the statistics
//   CTAs) each take a contiguous range of tiles per sweep (rotated by one CTA per sweep, so
//   that the longer ranges move around):
//     warp 0      W2 (B operand) TMA producer, two 64 KB stages, evict-last (W2 stays in L2);
//     warp 1      tensor-memory allocator and single-thread tcgen05.mma issuer (A from tensor
//                 memory: two slots, one per sweep parity);
//     warp 2      U TMA producer, two 32 KB stages, evict-first;
//     warps 4-11  epilogue: softmax partials (max, sum exp, first argmax) per 64 columns and,
//                 per row and column half, their merge over the CTA's range (the coarse
//                 partials); then the release of the sweep (counter `done`);
//     warps 12-15 the A operand of each sweep into tensor memory, once the group's previous
//                 tokens are drawn (counter `drawn`).
//   select CTAs run four 128-thread teams, one per row of a group: after every streaming CTA
//   released a sweep, a team draws its row's token with a two-level search (the row's coarse
//   partials, in vocabulary order, give the normaliser and the crossing tile range; that range's
//   64-column partials give the crossing segment, rebuilt element by element). The selects run
//   on SMs of their own (a quarter of the SMs, at most 32): on the streaming SMs they shared
//   issue slots with the epilogue warps and took several times longer.
//   target-statistics CTAs (only with a target rows pointer: 29 % of the SMs) stream the target
//   rows in 16 KB chunks through twelve bulk-copy stages into their softmax normalisers; they
//   share nothing with the proposal but the launch, and fill the time its serial chain leaves.
// Inter-CTA counters live at a fixed place of the caller's workspace; they are zero before a
// launch (workspace initialisation) and the last CTA to finish puts them back to zero. Every
// wait is bounded: on expiry the CTA sets SPEC_DEV_TIMEOUT and a workspace abort word, and
// every CTA then winds down, drains its copies and MMAs, frees its tensor memory and returns.
// The partials are those of the per-position tcgen05 pass; the draws are the same inverse-CDF
// rule with a two-level search, so they agree with the oracle to the same tolerances.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "select.cuh"
#include "tc_ptx.cuh"

namespace spec {
namespace prop {
using namespace tc;

constexpr int kBM = 128;                            // rows per group (TMEM lanes)
constexpr int kBN = 128;                            // vocabulary columns per tile
constexpr int kSeg = 64;                            // columns per partial
constexpr int kThreads = 512;
constexpr int kFirstEpi = 4, kEpiWarps = 8;
constexpr int kFirstSel = 12, kSelThreads = 128;
constexpr uint32_t kBoxBytes = kBM * 128;           // TMA box: 128 rows x 64 bf16
constexpr uint32_t kBAtomBytes = kBN * 128;         // 128 W2 rows x 64 K
constexpr uint32_t kBStageBytes = 4 * kBAtomBytes;  // K <= 256
constexpr uint32_t kUTileBytes = 2 * kBoxBytes;     // 128 rows x 128 columns
constexpr int kBStages = 2, kUStages = 2, kAccStages = 2;
constexpr int kAccCols = kAccStages * kBN;          // fp32 accumulators
constexpr int kACols = 128;                         // one A slot (rank <= 256)
constexpr int kTmemCols = 512;
static_assert(kAccCols + 2 * kACols <= kTmemCols, "tensor memory budget");
constexpr uint32_t kScratchBytes = 4096;            // per select warp: A-gather transpose
// The select stages each lane's run of partials (one float2 per 64-column segment) in the same
// 16 KB, so a row has at most 2048 segments (V <= 131072).
constexpr int kMaxSeg = 4 * kScratchBytes / 8;
constexpr int kSelBar = 1;                          // named barrier of the select warpgroup
constexpr int kMaxGrid = kMaxPropGrid;              // CTAs (tile ranges) a select covers
// target-statistics CTAs: rows in chunks of 8192 bf16 (16 KB) through 12 bulk-copy stages; one
// producer warp and one consumer warp per stage (chunk q: stage and warp q % 12, so that every
// wait on a stage's barrier is at most one phase ahead of it), a ring of row slots for the
// per-chunk partials
constexpr int kTChunk = 8192;
constexpr int kTStages = 12;
constexpr int kTConsumers = kTStages;
constexpr int kTParts = 32;  // chunks per row at most (V <= 262144)
constexpr int kTSlots = 8;

struct Params {
  RowJob j;        // rows = R, MAP_POSITION, MODE_STATS (k unused: each sweep has its own)
  SelectOut o;     // kind 0; the uniform of row r at position k is uni[r * gamma + k - 1]
  float* pm;       // [R, nseg] partials
  float* ps;
  int* pi;
  // coarse partials [R, grid, 2]: entry (r, c, h) merges row r's partials of column half h
  // over tile range c (the range a CTA takes in that sweep; ranges are in vocabulary order)
  float* cm;
  float* cs;
  int* ci;
  int nseg;        // 64-column partials per row
  int G;           // groups of up to 128 requests
  int ns;          // streaming CTAs (blocks 0 .. ns-1): tile ranges, partials, A gathers
  int nsel;        // select CTAs (blocks ns .. ns+nsel-1): four 128-thread select teams each
  int nstat;       // target-statistics CTAs (the rest; 0 without a target)
  // target rows [trows, V] whose softmax normalisers (m, log Z) of z = x * tscale go to
  // tstats [trows, 2] (independent of the proposal; fills the HBM time the proposal leaves)
  const void* T;
  float* tstats;
  int trows;
  float tscale;
  int n_nt;        // 128-column tiles
  int S;           // sweeps = gamma * G
  uint32_t* sync;  // done[S], drawn[S], exit count, abort word
  int stall;       // test of the bounded waits: the first W2 tile is never loaded
  int w1_32;       // W1 is 32-byte aligned: the A gather may use 32-byte loads
};

struct Smem {
  uint64_t b_full[kBStages], b_empty[kBStages];
  uint64_t u_full[kUStages], u_empty[kUStages];
  uint64_t acc_full[kAccStages], acc_empty[kAccStages];
  uint64_t a_full[2], a_empty[2];
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
  int flag;        // select warpgroup: broadcast of a wait's result
  int last;        // this CTA finished last
  int epi_prog[kEpiWarps];  // sweeps each epilogue warp has finished
  int released;              // sweeps this CTA has counted in `done`
};

// Shared memory of a target-statistics CTA (at the start of its dynamic shared memory).
struct StatSmem {
  unsigned char stage[kTStages][kTChunk * 2];
  uint64_t full[kTStages], empty[kTStages];
  float pm[kTSlots][kTParts];
  float ps[kTSlots][kTParts];
  int cnt[kTSlots];
};

// Shared memory of a select CTA (at the start of its dynamic shared memory).
struct SelSmem {
  SelectShared sel[4];
  uint4 w1s[4][32];  // each team's staged W1 row
  int flag[4];
  int abort;
  int last;
};

constexpr size_t kSmemBytes = 1024 + kBStages * kBStageBytes + kUStages * kUTileBytes +
                              4 * kScratchBytes + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "shared-memory budget");
static_assert(sizeof(StatSmem) + 1024 <= kSmemBytes - sizeof(Smem), "statistics CTA layout");

// Index of the tile range this streaming CTA takes in sweep s (the ranges rotate by one CTA per
// sweep, so that the longer ranges move around); ns ranges in vocabulary order.
__device__ __forceinline__ int range_index(int s, int ns) {
  return (int)(((long long)blockIdx.x + s) % ns);
}

// Tiles [tb, te) of tile range c.
__device__ __forceinline__ void range_tiles(int c, int ns, int n_nt, int& tb, int& te) {
  tb = (int)((long long)n_nt * c / ns);
  te = (int)((long long)n_nt * (c + 1) / ns);
}

// Tiles [tb, te) of sweep s for this streaming CTA.
__device__ __forceinline__ void sweep_range(int s, int ns, int n_nt, int& tb, int& te) {
  range_tiles(range_index(s, ns), ns, n_nt, tb, te);
}

// 1-D bulk copy global -> shared (16-byte aligned, a multiple of 16 bytes), completing on bar.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Draft logits of columns [v0, v0 + n) (n <= 64) by the 128 threads of a select team, with the
// previous token's W1 row staged in shared memory (w1s, rank / 8 chunks of 16 bytes): two
// threads per column, thread `part` summing chunks part, part + 2, ... of the rank-256 dot
// product in four independent chains, every W2 load of a thread in flight at once.
__device__ __forceinline__ void rebuild_segment(const RowJob& j, const RowInfo& ri,
                                                const uint4* w1s, int v0, int n, float* zs,
                                                int tid, NamedBarrier wg) {
  const int col = tid >> 1, part = tid & 1, v = v0 + col;
  const int nc = j.rank / 8;  // 16-byte chunks of a weight row (<= 32)
  float acc4[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // independent chains, summed at the end
  const float uval = col < n && part == 0 ? ld_elem<SPEC_BF16>(j.U, (size_t)ri.urow * j.V + v)
                                          : 0.0f;
  if (col < n) {
    const uint4* w2 = reinterpret_cast<const uint4*>(
        reinterpret_cast<const unsigned short*>(j.W2) + (size_t)v * j.rank);
    uint4 b[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int c = part + 2 * q;
      b[q] = c < nc ? __ldg(w2 + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int c = part + 2 * q;
      if (c < nc) {
        const uint4 a = w1s[c];
        const uint32_t aa[4] = {a.x, a.y, a.z, a.w};
        const uint32_t bb[4] = {b[q].x, b[q].y, b[q].z, b[q].w};
        float& acc = acc4[q & 3];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc = fmaf(__uint_as_float(aa[e] << 16), __uint_as_float(bb[e] << 16), acc);
          acc = fmaf(__uint_as_float(aa[e] & 0xffff0000u), __uint_as_float(bb[e] & 0xffff0000u),
                     acc);
        }
      }
    }
  }
  float acc = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  if (col < n && part == 0) {
    const float s = __fadd_rn(uval, acc);
    zs[col] = draft_allowed(j, ri.r, v) ? __fmul_rn(s, j.scale) : -INFINITY;
  }
  wg();
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One thread: bounded wait until *ctr >= target. On expiry, or when another CTA aborted, the
// local abort flag is raised (and, on expiry, the workspace abort word and SPEC_DEV_TIMEOUT).
__device__ bool spin_count(const uint32_t* ctr, uint32_t target, uint32_t* gabort,
                           volatile int* labort, uint32_t* status) {
  const long long t0 = clock64();
  while (true) {
    if (ld_acquire(ctr) >= target) return true;
    if (*labort) {
      atomicExch(gabort, 1u);
      return false;
    }
    if (*reinterpret_cast<volatile uint32_t*>(gabort)) {
      *labort = 1;
      return false;
    }
    if (clock64() - t0 > kSpinCycles) {
      *labort = 1;
      atomicExch(gabort, 1u);
      atomicOr(status, SPEC_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(20);
  }
}

// Two-level select of request r at position k (sweep s) by the 128 threads of the select
// warpgroup ("[DeepSeek-6] DSpark", section 3: x_k ~ softmax(U_k + W1[x_{k-1}] W2), or its
// argmax when greedy). Level 1: the 2 * grid coarse partials of the row give the maximum M, the
// normaliser Z (double-float sums of the range weights, in vocabulary order) and the tile range
// in which the cumulative mass first exceeds u * Z. Level 2: that range's 64-column partials
// give the crossing segment, which is rebuilt element by element (the rank-256 bias on CUDA
// cores) for the in-segment draw. The greedy token is the coarse partials' first maximum.
template <bool ARGMAX>
__device__ void select_two_level(const Params& P, const RowInfo& ri, int r, int s, int tid,
                                 NamedBarrier wg, SelectShared& S, uint4* w1s, uint32_t* drawn) {
  const RowJob& j = P.j;
  // loads that do not depend on the partials go out first: the previous token's W1 row (for the
  // segment rebuild) and the row's uniform
  if (tid < j.rank / 8)
    w1s[tid] = __ldg(reinterpret_cast<const uint4*>(j.W1) + (size_t)ri.prev * (j.rank / 8) + tid);
  const int grid = P.ns;  // tile ranges
  const int warp = tid >> 5, lane = tid & 31;
  const bool greedy = P.o.greedy != 0;
  const float u_row = greedy ? 0.0f : __ldg(P.o.uni + ri.urow);
  const size_t cb = (size_t)r * grid * 2;
  if (tid == 0) {
    S.c = -1;
    S.rem = 1e30f;
    S.x = -1;
    S.last = -1;
    S.zv0 = -1;
  }

  // level 1: ranges c = tid and tid + 128 (grid <= 256), both halves of each
  float em[2][2], es[2][2];
  float lmax = -INFINITY;
  int lidx = 0x7fffffff;
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    const int c = tid + 128 * a;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      em[a][h] = -INFINITY;
      es[a][h] = 0.0f;
      if (c < grid) {
        em[a][h] = __ldcg(P.cm + cb + 2 * c + h);
        es[a][h] = __ldcg(P.cs + cb + 2 * c + h);
        const int ix = ARGMAX ? __ldcg(P.ci + cb + 2 * c + h) : 0x7fffffff;
        if (em[a][h] > lmax || (em[a][h] == lmax && ix < lidx)) {
          lmax = em[a][h];
          lidx = ix;
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, lmax, off);
    const int oi = __shfl_xor_sync(0xffffffffu, lidx, off);
    if (om > lmax || (om == lmax && oi < lidx)) {
      lmax = om;
      lidx = oi;
    }
  }
  if (lane == 0) {
    S.wm[warp] = lmax;
    S.wi[warp] = lidx;
  }
  wg();
  float M = -INFINITY;
  int gidx = 0x7fffffff;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    if (S.wm[w] > M || (S.wm[w] == M && S.wi[w] < gidx)) {
      M = S.wm[w];
      gidx = S.wi[w];
    }
  }
  // range weights (the share of Z of each tile range), double-float; inclusive warp scans of
  // the ranges below 128 and of the others, and the warp totals in order
  auto weight = [&](float m, float sv) -> float {
    return sv == 0.0f ? 0.0f : sv * exp_shift(m, M);
  };
  DF wr[2], incl[2], before_lane[2];
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    wr[a] = df_add(DF{weight(em[a][0], es[a][0]), 0.0f}, weight(em[a][1], es[a][1]));
    incl[a] = warp_scan_df(wr[a]);
    before_lane[a] = df_shfl_up(incl[a], 1);
    if (lane == 0) before_lane[a] = df_zero();
    if (lane == 31) S.wt[4 * a + warp] = incl[a];
  }
  wg();
  // the eight warp totals in range order, scanned across lanes 0..7 of every warp (each warp
  // computes the same prefix sums): Z, and the mass before each warp's ranges
  DF pre = lane < 8 ? S.wt[lane] : df_zero();
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) {
    const DF y = df_shfl_up(pre, off);
    if (lane >= off && lane < 8) pre = df_add(y, pre);
  }
  const DF Z = df_shfl(pre, 7);
  if (tid == 0) {
    S.M = M;
    const bool zok = Z.hi > 0.0f && isfinite(Z.hi);
    S.lz = zok ? df_log(Z) : logf(Z.hi);
    if (!zok || !(M > -INFINITY)) atomicOr(j.status, SPEC_DEV_NONFINITE);
  }

  // the segment to rebuild: the greedy token's (for its log-probability) or the crossing one
  int x = -1;
  if (greedy) {
    x = gidx;
    if (x < 0 || x >= j.V) {
      if (tid == 0) atomicOr(j.status, SPEC_DEV_NONFINITE);
      x = 0;
    }
    if (tid == 0) {
      // the greedy token is known before its log-probability: publish it now
      P.o.tokens[ri.urow] = x;
      red_release_add(drawn, 1u);
      if (P.o.logp) S.zv0 = (x / kSeg) * kSeg;
    }
  } else {
    const DF t = df_mul(Z, u_row);
    // the crossing range: the warp (in range order) whose mass holds t, then its lane
    const unsigned wh = __ballot_sync(0xffffffffu, lane < 8 && df_gt(pre, t));
    const int wstar = wh ? __ffs(wh) - 1 : -1;
    const DF pb = df_shfl(pre, wstar > 0 ? wstar - 1 : 0);
    const DF before = wstar > 0 ? pb : df_zero();
    if (wstar >= 0 && warp == (wstar & 3)) {
      const int a = wstar >> 2;
      const DF ia = a ? incl[1] : incl[0], ba = a ? before_lane[1] : before_lane[0];
      const unsigned hit = __ballot_sync(0xffffffffu, df_gt(df_add(before, ia), t));
      if (hit && lane == __ffs(hit) - 1) {
        S.c = 128 * a + 32 * warp + lane;
        S.rem = df_float(df_add(t, df_neg(df_add(before, ba))));
      }
    }
    wg();
    if (S.c < 0 && tid == 0) {
      // rounding left no crossing: the last range with positive mass, drawn at its end
      int last = -1;
      for (int c = grid - 1; c >= 0 && last < 0; --c)
        if (__ldcg(P.cs + cb + 2 * c) > 0.0f || __ldcg(P.cs + cb + 2 * c + 1) > 0.0f) last = c;
      if (last < 0) atomicOr(j.status, SPEC_DEV_NONFINITE);
      S.c = last;
      S.rem = 1e30f;
    }
    wg();
    // level 2 (warp 0): the range's 64-column partials in vocabulary order, segment 2t + h for
    // tile t of the range and column half h; segments past V were never written and weigh 0
    const int cstar = S.c;
    if (warp == 0 && cstar >= 0) {
      int tb, te;
      range_tiles(cstar, P.ns, P.n_nt, tb, te);
      const int nf = 2 * (te - tb), sbase = 2 * tb;
      const float rem = S.rem;
      DF cum = df_zero();
      int found = -1, lastpos = -1;
      float rem2 = 1e30f;
      for (int b0 = 0; b0 < nf && found < 0; b0 += 32) {
        const int sg = sbase + b0 + lane;
        float wv = 0.0f;
        if (b0 + lane < nf && sg * kSeg < j.V) {
          const size_t o = (size_t)r * P.nseg + sg;
          wv = weight(__ldcg(P.pm + o), __ldcg(P.ps + o));
        }
        const DF inc = df_add(cum, warp_scan_df(DF{wv, 0.0f}));
        DF exc = df_shfl_up(inc, 1);
        if (lane == 0) exc = cum;
        const unsigned hit = __ballot_sync(0xffffffffu, df_gt(inc, DF{rem, 0.0f}));
        const unsigned pos = __ballot_sync(0xffffffffu, wv > 0.0f);
        if (pos) lastpos = sbase + b0 + 31 - __clz(pos);
        if (hit) {
          const int l = __ffs(hit) - 1;
          found = sbase + b0 + l;
          const DF e = df_shfl(exc, l);
          rem2 = df_float(df_add(DF{rem, 0.0f}, df_neg(e)));
        }
        cum = df_shfl(inc, 31);
      }
      if (lane == 0) {
        S.zv0 = (found >= 0 ? found : lastpos) * kSeg;  // segment start, or < 0
        S.rem = found >= 0 ? rem2 : 1e30f;
      }
    }
  }
  wg();
  // the segment's draft logits, element by element (one call site: two made the compiler run
  // out of registers)
  const int v0 = S.zv0;
  if (v0 >= 0) {
    const int n = min(kSeg, j.V - v0);
    rebuild_segment(j, ri, w1s, v0, n, S.zs, tid, wg);
    if (!greedy) {
      // exp(z - M) in token order; the first column whose running sum exceeds the remainder
      // (or the last one with mass)
      if (tid < n) S.es[tid] = exp_shift(S.zs[tid], M);
      wg();
      if (tid < 32) {
        const float rem = S.rem;
        const float a0 = tid < n ? S.es[tid] : 0.0f, a1 = tid + 32 < n ? S.es[tid + 32] : 0.0f;
        float s0 = a0, s1 = a1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y0 = __shfl_up_sync(0xffffffffu, s0, off);
          const float y1 = __shfl_up_sync(0xffffffffu, s1, off);
          if (tid >= off) {
            s0 += y0;
            s1 += y1;
          }
        }
        s1 += __shfl_sync(0xffffffffu, s0, 31);
        const unsigned m0 = __ballot_sync(0xffffffffu, s0 > rem && tid < n);
        const unsigned m1 = __ballot_sync(0xffffffffu, s1 > rem && tid + 32 < n);
        const unsigned p0 = __ballot_sync(0xffffffffu, a0 > 0.0f);
        const unsigned p1 = __ballot_sync(0xffffffffu, a1 > 0.0f);
        if (tid == 0) {
          if (m0) S.x = v0 + __ffs(m0) - 1;
          else if (m1) S.x = v0 + 32 + __ffs(m1) - 1;
          S.last = p1 ? v0 + 32 + 31 - __clz(p1) : (p0 ? v0 + 31 - __clz(p0) : -1);
        }
      }
    }
  }
  wg();
  if (!greedy) {
    x = S.x >= 0 ? S.x : S.last;
    if (x < 0) x = 0;  // no mass at all: the status word already records it
  }

  // outputs: the token first, counted at once (the gathers wait for it), then the rest
  const size_t q = (size_t)ri.urow;
  if (tid == 0 && !greedy) {
    P.o.tokens[q] = x;
    red_release_add(drawn, 1u);  // the token is visible before the count
  } else if (tid == 32) {
    if (P.o.w1) l2_prefetch_bytes(static_cast<const char*>(P.o.w1) + (size_t)x * P.o.w1_row_bytes,
                                  P.o.w1_row_bytes);
    if (P.o.logp) {
      const int zv0 = S.zv0;
      const bool in_seg = zv0 >= 0 && x >= zv0 && x < zv0 + kSeg;
      P.o.logp[q] = in_seg ? S.zs[x - zv0] - S.M - S.lz : -INFINITY;
    }
    if (P.o.stats) {
      P.o.stats[2 * q] = S.M;
      P.o.stats[2 * q + 1] = S.lz;
    }
  }
}

template <bool ARGMAX>
__global__ void __launch_bounds__(kThreads, 1)
    markov_propose_kernel(const __grid_constant__ CUtensorMap map_w2,
                          const __grid_constant__ CUtensorMap map_u, const __grid_constant__ Params P) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sB = smem;
  unsigned char* sU = sB + kBStages * kBStageBytes;
  unsigned char* sScr = sU + kUStages * kUTileBytes;
  Smem& sh = *reinterpret_cast<Smem*>(sScr + 4 * kScratchBytes);
  volatile int* abort = &sh.abort;

  const RowJob& j = P.j;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* status = j.status;
  const int S = P.S, G = P.G;
  uint32_t* done = P.sync;
  uint32_t* drawn = P.sync + S;
  uint32_t* exitc = P.sync + 2 * S;
  uint32_t* gabort = P.sync + 2 * S + 1;
  const int ka_n = j.rank / 64;

  if (blockIdx.x >= P.ns + P.nsel) {
    // ================================================================ target-statistics CTA
    // A contiguous block of target rows; each 8192-column chunk is reduced by one warp to
    // (max z, sum exp(z - max)), z = x * tscale, and the warp that completes a row's chunks
    // merges them in chunk order into (m, log Z).
    StatSmem& st = *reinterpret_cast<StatSmem*>(smem);
    const int c = blockIdx.x - P.ns - P.nsel;
    const int rb = (int)((long long)P.trows * c / P.nstat);
    const int re = (int)((long long)P.trows * (c + 1) / P.nstat);
    const int parts = (j.V + kTChunk - 1) / kTChunk;
    const long long nq = (long long)(re - rb) * parts;
    if (threadIdx.x == 0) {
      for (int x = 0; x < kTStages; ++x) {
        mbar_init(&st.full[x], 1);
        mbar_init(&st.empty[x], 1);
      }
      for (int x = 0; x < kTSlots; ++x) st.cnt[x] = 0;
      sh.abort = 0;
      sh.last = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const unsigned short* Tb = static_cast<const unsigned short*>(P.T);
    if (warp == 0) {
      // producer: chunk q into stage q % kTStages once its previous chunk is consumed
      if (lane == 0) {
        const uint64_t pol = policy_evict_first();
        long long q = 0;
        for (; q < nq; ++q) {
          const int x = (int)(q % kTStages);
          const uint32_t ph = (uint32_t)((q / kTStages) & 1);
          if (!mbar_wait(&st.empty[x], ph ^ 1, abort, status)) break;
          const int row = rb + (int)(q / parts), part = (int)(q % parts);
          const int n0 = part * kTChunk, n = min(kTChunk, j.V - n0);
          mbar_arrive_expect_tx(&st.full[x], (uint32_t)n * 2);
          bulk_load(st.stage[x], Tb + (size_t)row * j.V + n0, (uint32_t)n * 2, &st.full[x], pol);
        }
        // every issued copy lands before the CTA moves on
        for (long long d = q > kTStages ? q - kTStages : 0; d < q; ++d)
          mbar_drain(&st.full[d % kTStages], (uint32_t)((d / kTStages) & 1));
      }
    } else if (warp <= kTConsumers) {
      const int cw = warp - 1;  // consumes stage cw: chunks cw, cw + kTStages, ...
      for (long long q = cw; q < nq; q += kTConsumers) {
        const int x = (int)(q % kTStages);
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&st.full[x], (uint32_t)((q / kTStages) & 1), abort, status)))
          break;
        const int ri = (int)(q / parts), part = (int)(q % parts);
        const int nw = min(kTChunk, j.V - part * kTChunk) / 8;  // 16-byte words
        const uint32_t base = smem_u32(st.stage[x]);
        // one pass: batches of four words per lane, the running maximum of the raw values (the
        // scale is positive) with at most one rescale per batch, exp2((x - max) * scale * log2e)
        // in packed pairs; padding words decode to -inf
        const float cl = P.tscale * kLog2e;
        float mx = -INFINITY;
        unsigned long long s2 = pack2(0.0f, 0.0f);
        for (int w0 = lane; w0 < nw; w0 += 4 * 32) {
          float xv[4][8];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int w = w0 + 32 * b;
            const uint4 v = w < nw ? lds128(base + w * 16)
                                   : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
            unpack_bf16x8(v, xv[b]);
          }
          float g = mx;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            g = fmaxf(g, max3(max3(xv[b][0], xv[b][1], xv[b][2]), max3(xv[b][3], xv[b][4], xv[b][5]),
                              fmaxf(xv[b][6], xv[b][7])));
          if (g > mx) {
            if (mx > -INFINITY) {
              const float f = fast_exp2((mx - g) * cl);
              s2 = mul2(s2, pack2(f, f));
            }
            mx = g;
          }
          if (mx > -INFINITY) {
            const unsigned long long nm = pack2(-mx, -mx), c2 = pack2(cl, cl);
#pragma unroll
            for (int b = 0; b < 4; ++b)
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                float a0, a1;
                unpack2(mul2(add2(pack2(xv[b][e], xv[b][e + 1]), nm), c2), a0, a1);
                s2 = add2(s2, pack2(fast_exp2(a0), fast_exp2(a1)));
              }
          }
        }
        float sa, sb;
        unpack2(s2, sa, sb);
        // merge the lanes in the scaled domain: (m = max * scale, s)
        const StatsAcc acc = warp_merge(
            StatsAcc{mx > -INFINITY ? __fmul_rn(mx, P.tscale) : -INFINITY, sa + sb, 0});
        const float m = acc.m, sum = acc.s;
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&st.empty[x]);  // the stage may be refilled
          const int slot = ri % kTSlots;
          st.pm[slot][part] = m;
          st.ps[slot][part] = sum;
          __threadfence_block();
          if (atomicAdd(&st.cnt[slot], 1) == parts - 1) {
            // the row's last chunk: merge its chunks in order
            __threadfence_block();
            const volatile float* vm = st.pm[slot];
            const volatile float* vs = st.ps[slot];
            StatsAcc a = stats_empty();
            for (int pp = 0; pp < parts; ++pp) a = stats_merge(a, StatsAcc{vm[pp], vs[pp], 0});
            st.cnt[slot] = 0;
            const size_t row = (size_t)(rb + ri);
            P.tstats[2 * row] = a.m;
            P.tstats[2 * row + 1] = logf(a.s);
            if (!(a.m > -INFINITY) || !(a.s > 0.0f) || !isfinite(a.s))
              atomicOr(status, SPEC_DEV_NONFINITE);
          }
        }
      }
    }
  } else if (blockIdx.x >= P.ns) {
    // ================================================================ select CTA
    // Four teams of four warps; team T of all select CTAs draws rows T, T + 4 nsel, ... of
    // every group, once every streaming CTA released the sweep.
    SelSmem& ss = *reinterpret_cast<SelSmem*>(smem);
    if (threadIdx.x == 0) {
      sh.abort = 0;
      sh.last = 0;
    }
    __syncthreads();
    const int team = warp >> 2, tid = threadIdx.x & 127;
    const NamedBarrier tbar{1 + team, kSelThreads};
    const int T = (blockIdx.x - P.ns) * 4 + team, nteams = P.nsel * 4;
    bool ok = true;
    for (int s = 0; s < S && ok; ++s) {
      const int g = s % G, k = s / G + 1;
      const int rows_g = min(kBM, j.R - g * kBM);
      if (T >= rows_g) continue;
      if (tid == 0) ss.flag[team] = spin_count(&done[s], P.ns, gabort, abort, status) ? 1 : 0;
      tbar();
      ok = ss.flag[team] != 0;
      tbar();
      if (!ok) break;
      for (int ig = T; ig < rows_g; ig += nteams) {
        const int r = g * kBM + ig;
        RowInfo ri;
        ri.active = 1;
        ri.r = r;
        ri.urow = (long long)r * j.gamma + (k - 1);
        ri.trow = -1;
        ri.resid = 0;
        int p = k == 1 ? j.anchors[r] : __ldcg(j.tokens + (size_t)r * j.gamma + k - 2);
        if (p < 0 || p >= j.V) {
          if (tid == 0) atomicOr(status, SPEC_DEV_BAD_TOKEN);
          p = 0;
        }
        ri.prev = p;
        select_two_level<ARGMAX>(P, ri, r, s, tid, tbar, ss.sel[team], ss.w1s[team], &drawn[s]);
        tbar();
      }
    }
    if (!ok) *abort = 1;
  } else {
  // ================================================================ streaming CTA
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&sh.b_full[s], 1);
      mbar_init(&sh.b_empty[s], 1);
    }
    for (int s = 0; s < kUStages; ++s) {
      mbar_init(&sh.u_full[s], 1);
      mbar_init(&sh.u_empty[s], kEpiWarps);
    }
    for (int s = 0; s < kAccStages; ++s) {
      mbar_init(&sh.acc_full[s], 1);
      mbar_init(&sh.acc_empty[s], kEpiWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.a_full[s], 1);
      mbar_init(&sh.a_empty[s], 1);
    }
    mbar_init(&sh.drain, 1);
    sh.abort = 0;
    sh.flag = 0;
    sh.last = 0;
    for (int w = 0; w < kEpiWarps; ++w) sh.epi_prog[w] = 0;
    sh.released = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sh.tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_slot;

  if (warp < kFirstEpi) {
    if (warp == 0) {
      // ---------------------------------------------------------------- W2 (B) producer
      const uint64_t pol_keep = policy_evict_last();
      int bs = 0;
      uint32_t bph = 0;
      bool ok = true, first = true;
      for (int s = 0; s < S && ok; ++s) {
        int tb, te;
        sweep_range(s, P.ns, P.n_nt, tb, te);
        for (int t = tb; t < te && ok; ++t) {
          ok = mbar_wait(&sh.b_empty[bs], bph ^ 1, abort, status);
          if (ok && lane == 0 && !(P.stall && first)) {
            mbar_arrive_expect_tx(&sh.b_full[bs], ka_n * kBAtomBytes);
            for (int ka = 0; ka < ka_n; ++ka)
              tma_load_2d(sB + bs * kBStageBytes + ka * kBAtomBytes, &map_w2, ka * 64, t * kBN,
                          &sh.b_full[bs], pol_keep);
          }
          first = false;
          if (++bs == kBStages) { bs = 0; bph ^= 1; }
        }
      }
      if (lane == 0)
        for (int s = 0; s < kBStages; ++s) mbar_drain(&sh.b_full[s], (s < bs) ? bph : (bph ^ 1));
    } else if (warp == 2) {
      // ---------------------------------------------------------------- U producer
      const uint64_t pol_stream = policy_evict_first();
      int us = 0;
      uint32_t uph = 0;
      bool ok = true;
      for (int s = 0; s < S && ok; ++s) {
        const int g = s % G, k = s / G + 1;
        int tb, te;
        sweep_range(s, P.ns, P.n_nt, tb, te);
        for (int t = tb; t < te && ok; ++t) {
          ok = mbar_wait(&sh.u_empty[us], uph ^ 1, abort, status);
          if (ok && lane == 0) {
            unsigned char* du = sU + us * kUTileBytes;
            mbar_arrive_expect_tx(&sh.u_full[us], kUTileBytes);
            for (int b = 0; b < 2; ++b)
              tma_load_3d(du + b * kBoxBytes, &map_u, t * kBN + b * 64, k - 1, g * kBM,
                          &sh.u_full[us], pol_stream);
          }
          if (++us == kUStages) { us = 0; uph ^= 1; }
        }
      }
      if (lane == 0)
        for (int s = 0; s < kUStages; ++s) mbar_drain(&sh.u_full[s], (s < us) ? uph : (uph ^ 1));
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16(kBM, kBN);
      if (lane == 0) {
        bool ok = true;
        int bs = 0, as = 0;
        uint32_t bph = 0;
        uint32_t accph[kAccStages] = {};
        for (int s = 0; s < S && ok; ++s) {
          const int slot = s & 1;
          ok = mbar_wait(&sh.a_full[slot], (s >> 1) & 1, abort, status);
          if (!ok) break;
          tc_fence_after();
          int tb, te;
          sweep_range(s, P.ns, P.n_nt, tb, te);
          for (int t = tb; t < te && ok; ++t) {
            ok = mbar_wait(&sh.b_full[bs], bph, abort, status);
            if (!ok) break;
            tc_fence_after();
            ok = mbar_wait(&sh.acc_empty[as], accph[as] ^ 1, abort, status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d = tmem + as * kBN;
            const uint32_t a = tmem + kAccCols + slot * kACols;
            for (int ka = 0; ka < ka_n; ++ka) {
              const uint32_t b_base = smem_u32(sB + bs * kBStageBytes + ka * kBAtomBytes);
              // K = 16 per instruction: 8 tensor-memory columns of A, 32 bytes of a B row
  #pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ta(d, a + ka * 32 + ks * 8, sw128_desc(b_base + ks * 32), idesc,
                            (ka | ks) != 0);
            }
            mma_commit(&sh.acc_full[as]);
            accph[as] ^= 1;
            if (++as == kAccStages) as = 0;
            mma_commit(&sh.b_empty[bs]);
            if (++bs == kBStages) { bs = 0; bph ^= 1; }
          }
          if (!ok) break;
          mma_commit(&sh.a_empty[slot]);  // the slot may be refilled once these MMAs complete
        }
        // all MMAs issued by this thread complete before tensor memory is released
        mma_commit(&sh.drain);
        mbar_drain(&sh.drain, 0);
      }
      __syncwarp();
    }
  } else if (warp < kFirstSel) {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - kFirstEpi;
    const int q = warp & 3;       // TMEM lane quarter
    const int h = ew >> 2;        // column half
    const int i = q * 32 + lane;  // row within the group (TMEM lane)
    const int col0 = h * kSeg;
    int as = 0, us = 0;
    uint32_t accph[kAccStages] = {}, uph = 0;
    bool ok = true;
    for (int s = 0; s < S && ok; ++s) {
      const int g = s % G;
      const int r = g * kBM + i;
      const bool valid = r < j.R;
      int tb, te;
      sweep_range(s, P.ns, P.n_nt, tb, te);
      StatsAcc coarse = stats_empty();  // this thread's half of the range, merged in order
      for (int t = tb; t < te && ok; ++t) {
        const int n0 = t * kBN;
        const bool live = valid && n0 + col0 < j.V;
        const bool tail = n0 + kBN > j.V;
        // allowed-token bits of this thread's columns (grammar-masked drafting), loaded before
        // the waits so that the load is in flight meanwhile
        uint32_t mlo = ~0u, mhi = ~0u;
        if (j.mask && live) {
          const uint32_t* mr = j.mask + (size_t)r * j.mask_words + ((n0 + col0) >> 5);
          mlo = mr[0];
          mhi = n0 + col0 + 32 < j.V ? mr[1] : 0u;
        }
        // every lane waits; the warp goes on only if all did (tcgen05.ld is warp-wide)
        ok = __all_sync(0xffffffffu, mbar_wait(&sh.acc_full[as], accph[as], abort, status));
        if (!ok) break;
        tc_fence_after();
        ok = __all_sync(0xffffffffu, mbar_wait(&sh.u_full[us], uph, abort, status));
        if (!ok) break;
        // TMEM reads and shared-memory reads first, then release the stages
        uint32_t braw[kSeg];
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + as * kBN + col0;
        tmem_ld32_async(taddr, braw);
        tmem_ld32_async(taddr + 32, braw + 32);
        const uint32_t u_base = smem_u32(sU + us * kUTileBytes);
        uint4 uw[kSeg / 8];
#pragma unroll
        for (int c = 0; c < kSeg / 8; ++c) {
          const int col = col0 + 8 * c;
          const int b = col >> 6, cc = (col & 63) >> 3;
          uw[c] = lds128(u_base + b * kBoxBytes + i * 128 + ((cc ^ (i & 7)) << 4));
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sh.acc_empty[as]);
          mbar_arrive(&sh.u_empty[us]);
        }
        if (++us == kUStages) { us = 0; uph ^= 1; }
        accph[as] ^= 1;
        if (++as == kAccStages) as = 0;
        float m, sum;
        int idx;
        stats_partial64<ARGMAX>(braw, uw, j.scale, n0 + col0, j.V, tail, j.mask != nullptr, mlo,
                                mhi, m, sum, idx);
        if (live) {
          const size_t o = (size_t)r * P.nseg + (n0 + col0) / kSeg;
          P.pm[o] = m;
          P.ps[o] = sum;
          if (ARGMAX) P.pi[o] = idx;
          coarse = stats_merge(coarse, StatsAcc{m, sum, idx});
        }
      }
      if (!ok) break;
      if (valid) {
        const size_t o = ((size_t)r * P.ns + range_index(s, P.ns)) * 2 + h;
        P.cm[o] = coarse.m;
        P.cs[o] = coarse.s;
        if (ARGMAX) P.ci[o] = coarse.idx;
      }
      // release: each thread's partials are visible before its warp records its progress;
      // the CTA has finished the sweeps below the slowest warp's progress, and whichever warp
      // raises that minimum counts them in `done` (no barrier, so a warp that stopped early
      // cannot hold the others, and a warp that runs sweeps ahead is not miscounted)
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        volatile int* prog = sh.epi_prog;
        prog[ew] = s + 1;
        __threadfence_block();
        int m = prog[0];
        for (int w = 1; w < kEpiWarps; ++w) m = min(m, prog[w]);
        const int from = atomicMax(&sh.released, m);
        for (int x = from; x < m; ++x) red_release_add(&done[x], 1u);
      }
    }
  } else {
    // ---------------------------------------------------------------- A gather
    const int tid = threadIdx.x - kFirstSel * 32;
    const int sq = warp & 3;  // TMEM lane quarter
    const NamedBarrier wg{kSelBar, kSelThreads};
    const uint32_t scr = smem_u32(sScr) + (warp - kFirstSel) * kScratchBytes;
    const uint4* w1 = reinterpret_cast<const uint4*>(j.W1);
    const int nch = j.rank / 8;  // 16-byte chunks of a W1 row (<= 32)

    // bounded wait of the warpgroup on an inter-CTA counter
    auto wait_count = [&](const uint32_t* ctr, uint32_t target) -> bool {
      if (tid == 0) sh.flag = spin_count(ctr, target, gabort, abort, status) ? 1 : 0;
      wg();
      const bool r = sh.flag != 0;
      wg();
      return r;
    };

    // A operand of sweep t: the W1 rows of the group's previous tokens into slot t % 2. The
    // rows are read whole (four lanes per 128-byte piece, eight rows per instruction) and turned
    // into one row per lane through the warp's 4 KB scratch.
    auto gather = [&](int t) -> bool {
      const int g = t % G, k = t / G + 1, slot = t & 1;
      const int rows_g = min(kBM, j.R - g * kBM);
      if (t >= G && !wait_count(&drawn[t - G], (uint32_t)rows_g)) return false;
      if (t >= 2) {  // one thread waits for the slot, the warpgroup follows its result
        if (tid == 0) sh.flag = mbar_wait(&sh.a_empty[slot], ((t - 2) >> 1) & 1, abort, status);
        wg();
        const bool free = sh.flag != 0;
        wg();
        if (!free) return false;
      }
      tc_fence_after();
      const int r = g * kBM + sq * 32 + lane;
      int prev = -1;
      if (r < j.R) {
        const int p = k == 1 ? j.anchors[r] : __ldcg(j.tokens + (size_t)r * j.gamma + k - 2);
        if (p < 0 || p >= j.V) atomicOr(status, SPEC_DEV_BAD_TOKEN);  // row read as zeros
        else prev = p;
      }
      const uint32_t a_addr = tmem + ((uint32_t)(sq * 32) << 16) + kAccCols + slot * kACols;
      const int npieces = (nch + 7) / 8;
      for (int p0 = 0; p0 < npieces; p0 += 2) {
        uint4 v[2][8];
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int rl = 8 * kk + (lane >> 2), c = 8 * (p0 + pp) + 2 * (lane & 3);
            const int row = __shfl_sync(0xffffffffu, prev, rl);
            uint4 a = make_uint4(0, 0, 0, 0), b = a;
            if (row >= 0 && c < nch) {  // nch is a multiple of 8, so chunk c + 1 is in the row
              const uint4* src = w1 + (size_t)row * nch + c;
              if (P.w1_32) {
                asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                             : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y),
                               "=r"(b.z), "=r"(b.w)
                             : "l"(src));
              } else {
                a = __ldg(src);
                b = __ldg(src + 1);
              }
            }
            v[pp][2 * kk] = a;
            v[pp][2 * kk + 1] = b;
          }
        }
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const int piece = p0 + pp;
          if (piece >= npieces) break;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int rl = 8 * kk + (lane >> 2), cc = 2 * (lane & 3);
            sts128(scr + rl * 128 + ((cc ^ (rl & 7)) << 4), v[pp][2 * kk]);
            sts128(scr + rl * 128 + (((cc + 1) ^ (rl & 7)) << 4), v[pp][2 * kk + 1]);
          }
          __syncwarp();
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 x = lds128(scr + lane * 128 + ((c ^ (lane & 7)) << 4));
            w[4 * c] = x.x;
            w[4 * c + 1] = x.y;
            w[4 * c + 2] = x.z;
            w[4 * c + 3] = x.w;
          }
          __syncwarp();
          // chunk c of the row holds K elements 8c..8c+7 = tensor-memory columns 4c..4c+3
          if (8 * piece < nch) tmem_st16(a_addr + 32 * piece, w);
          if (8 * piece + 4 < nch) tmem_st16(a_addr + 32 * piece + 16, w + 16);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      wg();
      if (tid == 0) mbar_arrive(&sh.a_full[slot]);
      return true;
    };

    // the A operands in sweep order (each waits for its group's previous draws and its slot)
    bool ok = true;
    for (int t = 0; t < S && ok; ++t) ok = gather(t);
    if (!ok) *abort = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  }  // streaming CTA
  // the last CTA to finish puts the counters back to zero for the next launch; a CTA that
  // stopped early tells the others first
  __syncthreads();
  if (threadIdx.x == 0) {
    if (sh.abort) atomicExch(gabort, 1u);
    __threadfence();
    sh.last = atomicAdd(exitc, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (sh.last) {
    __threadfence();
    for (int x = threadIdx.x; x < 2 * S + 2; x += blockDim.x) P.sync[x] = 0u;
  }
}

}  // namespace prop

bool markov_propose_tc_supported(int udt, int wdt, int rank, int R, int gamma, int V,
                                 const void* U, const void* W1, const void* W2) {
  if (R < 1 || gamma < 1) return false;
  if ((V + prop::kSeg - 1) / prop::kSeg > prop::kMaxSeg) return false;
  if (num_sms() > prop::kMaxGrid || num_sms() < 2) return false;
  const long long sweeps = (long long)gamma * ((R + prop::kBM - 1) / prop::kBM);
  if (2 * sweeps + 2 > (long long)(kSyncBytes / 4)) return false;
  return markov_tc_supported(udt, wdt, rank, V, U, nullptr, W1, W2);
}

cudaError_t launch_markov_propose_tc(const RowJob& j, const SelectOut& o, float* pm, float* ps,
                                     int* pi, bool argmax, uint32_t* sync, cudaStream_t s,
                                     const void* target, float* tstats, float tscale) {
  using namespace prop;
  TraceScope ts(SPEC_KCLASS_PROPOSE, s);
  Params p;
  memset(&p, 0, sizeof p);
  p.j = j;
  p.o = o;
  p.pm = pm;
  p.ps = ps;
  p.pi = pi;
  p.nseg = (j.V + kSeg - 1) / kSeg;
  // one CTA per SM: a quarter of them at most (32 at most, four teams each: one team per row
  // of a 128-row group) select, the others stream
  const int grid = num_sms();
  p.nsel = grid / 4 < 32 ? grid / 4 : 32;
  if (p.nsel < 1) p.nsel = 1;
  // with a target, 29 % of the SMs stream its rows for the normalisers meanwhile: a statistics
  // CTA reduces about 40 GB/s, and every CTA taken from the streaming ones lengthens the
  // proposal. At R = 256, gamma = 7 on 152 SMs the launch is shortest with 43-44 (305 us;
  // 310 us at 42 or 45, 321 us at 47, 354 us at 36 or 58)
  p.nstat = target ? grid * 29 / 100 : 0;
  if (target && p.nstat < 1) p.nstat = 1;
  p.ns = grid - p.nsel - p.nstat;
  if (p.ns < 1) return cudaErrorInvalidConfiguration;
  p.T = target;
  p.tstats = tstats;
  p.trows = target ? j.R * (j.gamma + 1) : 0;
  p.tscale = tscale;
  // the coarse partials follow the fine ones in the same arrays
  const size_t fine = (size_t)j.R * p.nseg;
  p.cm = pm + fine;
  p.cs = ps + fine;
  p.ci = pi ? pi + fine : nullptr;
  p.G = (j.R + kBM - 1) / kBM;
  p.n_nt = (j.V + kBN - 1) / kBN;
  p.S = j.gamma * p.G;
  p.sync = sync;
  p.stall = take_stall_request();
  p.w1_32 = (reinterpret_cast<uintptr_t>(j.W1) & 31) == 0;
  CUtensorMap w2, u;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)j.rank, (cuuint64_t)j.V};
    const cuuint64_t str[1] = {(cuuint64_t)j.rank * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBN};
    if (!make_tensor_map_bf16(&w2, j.W2, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kBM};
    const cuuint64_t du[3] = {(cuuint64_t)j.V, (cuuint64_t)j.gamma, (cuuint64_t)j.R};
    const cuuint64_t su[2] = {(cuuint64_t)j.V * 2, (cuuint64_t)j.V * 2 * j.gamma};
    if (!make_tensor_map_bf16(&u, j.U, 3, du, su, box)) return cudaErrorInvalidValue;
  }
  auto k = argmax ? markov_propose_kernel<true> : markov_propose_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  // one CTA per SM; every CTA must be resident at once (the counters are waited on)
  return launch_kernel(k, dim3(grid), dim3(kThreads), kSmemBytes, s, false, w2, u, p);
}

}  // namespace spec
