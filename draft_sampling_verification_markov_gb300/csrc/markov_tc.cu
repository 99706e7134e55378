// markov_tc.cu -- tcgen05 Markov producer: the rank-r bias GEMM W1[x_{k-1}] . W2^T on the
// 5th-generation tensor cores, fused with the per-row epilogue of each pass ("[DeepSeek-6]
// DSpark", section 4 "Markov Head": B(x_{k-1}, .) = W1[x_{k-1}] W2 added to the base logits,
// section 3 softmax; section 5 TV label; the residual of rejection sampling).
//
// One tile = 128 rows (requests, TMEM lanes) x N = 128 vocabulary columns, K = rank (<= 256, a
// multiple of 64). A work unit is one W2 column tile against a pair of row blocks: the B tile
// is loaded once and feeds both blocks' MMA groups, which halves the W2 bytes each SM pulls
// into shared memory.
//   A  [128 x rank] bf16 per row block: the W1 rows of each row's previous token, gathered by
//      the epilogue warps (the first pair of a CTA through a shared-memory transpose, so that
//      the rows are read whole) and stored into tensor memory with tcgen05.st (lane = row, two
//      bf16 of K per 32-bit column); both blocks of the current pair stay resident.
//   B  [N x rank] bf16: W2 rows (W2 stored [V, rank], K-major) by TMA, one whole tile per
//      pipeline stage, kept in L2 with an evict-last policy. W2 is re-read by every position
//      and stays in L2 while the logit streams are evict-first, so no copy is prefetched: an
//      L2 prefetch two units ahead, and one of all of W2 by the select kernel, only queued in
//      front of the copies the pipeline waits for.
//   D  [128 x N] fp32 in tensor memory (2 stages), read back with tcgen05.ld.
//   U / T tiles: the base-logit (and target) rows of each (unit, row block), by TMA with an
//      evict-first policy (read once), 64-column boxes in the 128-byte-swizzled layout; rows
//      that are not equally spaced (the final rows of rejection verification) are copied by
//      six copier warps with 16-byte cp.async into the same layout, each row's piece read
//      whole by neighbouring lanes.
// The W1 rows of the A gather are prefetched into L2 by the kernel that drew the tokens, so
// the logit stream starts at once.
// Warp roles (one CTA per SM, persistent over a contiguous range of units; struct Roles):
//   warp 0  W2 (B operand) TMA producer;  warp 1  TMEM allocator + single-thread MMA issuer;
//   tiles by TMA (384 threads): warp 2  U / T tile producer, warps 3..10  epilogue, warp 11
//   idle; gathered rows (512 threads): warps 2, 3 and 12..15  row copiers, warps 4..11
//   epilogue. An epilogue warp w reads TMEM lanes 32*(w%4).. and one column half of the tile.
// Epilogues (per row, per N/2-column half tile, one partial each):
//   MODE_STATS  z = (U + bias) * scale -> (max z, sum exp(z - max), first argmax);
//   MODE_TV     sum min(p_d, p_t);    MODE_RESID  sum max(0, p_t - p_d) (p_t on bonus rows).
// Every mbarrier wait is bounded (about a second); on expiry the CTA sets SPEC_DEV_TIMEOUT,
// drains its own copies and MMAs, frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace spec {
namespace tc {

constexpr int kBM = 128;                            // rows per tile (one MMA, 128 TMEM lanes)
constexpr int kEpiWarps = 8;

// Warp roles. Tiles by TMA (12 warps): 0 W2 producer, 1 MMA issuer, 2 U / T producer, 3..10
// epilogue, 11 idle. Gathered rows (16 warps): 0 W2 producer, 1 MMA issuer, 2, 3 and 12..15
// row copiers, 4..11 epilogue. A copier warp moves about 10 GB/s of 256-byte row pieces with
// cp.async, so the gathered rows need several; the copiers and producers (warpgroups 0 and 3)
// run on 80 registers and hand the rest to the epilogue warpgroups (1 and 2), which get 176:
// 4 x 128 threads x 128 registers at launch = 2 x 128 x 80 + 2 x 128 x 176.
template <bool GATHER>
struct Roles {
  static constexpr int kWarps = GATHER ? 16 : 12;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kFirstEpi = GATHER ? 4 : 3;
  static constexpr int kCopiers = GATHER ? 6 : 1;
  static constexpr int kRegsLow = 80, kRegsHigh = 176;
  static_assert(!GATHER || 2 * kRegsLow + 2 * kRegsHigh == 4 * (65536 / kThreads),
                "register split");
};
constexpr uint32_t kBoxBytes = kBM * 128;         // one TMA box: 128 rows x 64 columns (bf16)

// Per pass mode. Shared memory (A lives in tensor memory):
//   MODE_STATS:          B 2 x 64 KB + U 2 x 32 KB             = 192 KB; TMEM 2 x 128 + 2 x 128 cols
//   MODE_TV, MODE_RESID: B 1 x 64 KB + (U + T) 2 x 2 x 32 KB   = 192 KB; TMEM 2 x 128 + 2 x 128
// N = 128 columns everywhere. The pair passes read two logit tensors; a row piece of 256 bytes
// costs little more HBM time than one of 128 bytes, so they take the wide tile at the price of
// a single W2 stage (the TV pass went from 1.51 to 1.29 ms at R = 512, gamma = 16).
template <int MODE>
struct Cfg {
  static constexpr int kBN = 128;                             // vocabulary columns per tile
  static constexpr int kBoxes = kBN / 64;                     // 64-column boxes per logit tile
  static constexpr uint32_t kBAtomBytes = kBN * 128;          // kBN W2 rows x 64 K
  static constexpr uint32_t kBStageBytes = 4 * kBAtomBytes;   // K <= 256
  static constexpr int kBStages = MODE == MODE_STATS ? 2 : 1;
  static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;
  // two stages: a third kept more copies queued ahead of the W2 tile the MMA waits for
  static constexpr int kUStages = 2;
  static constexpr int kAccStages = kBN == 128 ? 2 : 4;       // accumulator stages in TMEM
  static constexpr int kAccCols = kAccStages * kBN;
  static constexpr int kACols = 128;                          // one A block (rank <= 256)
  static constexpr int kTmemCols = 512;                       // accumulators + two A blocks
  static_assert(kAccCols + 2 * kACols <= kTmemCols, "tensor memory budget");
  static constexpr int kSeg = kBN / 2;                        // columns per epilogue warp / partial
};

// ------------------------------------------------------------------------------ tiles

struct Tiles {
  int n_mt, n_nt;  // row blocks (128 rows) and column tiles
  int rb;          // row blocks per draft position (MAP_ALL_POS)
};

struct TileRow {
  int valid;
  int r;
  int k;      // draft position (1-based) of this row block (uniform modes)
  int prow;   // partial row index in the pass
};

// Row `i` (0..127) of row block mt.
__device__ __forceinline__ TileRow tile_row(const RowJob& j, const Tiles& t, int mt, int i) {
  TileRow o;
  if (j.map == MAP_ALL_POS) {
    o.k = mt / t.rb + 1;
    o.r = (mt % t.rb) * kBM + i;
    o.prow = o.r * j.gamma + (o.k - 1);
  } else {
    o.k = j.k;
    o.r = mt * kBM + i;
    o.prow = o.r;
  }
  o.valid = o.r < j.R;
  return o;
}

// ------------------------------------------------------------------------------ kernel

struct TcParams {
  RowJob j;
  Tiles t;
  float* pm;
  float* ps;
  int* pi;
  int nseg;   // partial segments per row (row-major partial arrays)
  int stall;  // test of the bounded waits: the first W2 tile is never loaded
  int w1_32;  // W1 is 32-byte aligned: the first A gather may use 32-byte loads
};

// Per-row normalisers of the pair modes for one row (loaded once per row block).
template <int MODE>
__device__ __forceinline__ void row_norms_tc(const RowJob& j, const TileRow& tr, Norm& dn,
                                             Norm& tn, bool& resid) {
  dn = {0.0f, 0.0f};
  tn = {0.0f, 0.0f};
  resid = true;
  if (!tr.valid) return;
  if constexpr (MODE == MODE_TV) {
    tn = load_norm(j.tstats, target_row(j, tr.r, tr.k - 1));
    dn = load_norm(j.dstats, (long long)tr.r * j.gamma + (tr.k - 1));
  } else {
    const int n = j.final_n[tr.r];
    resid = j.final_kind[tr.r] != 0;
    tn = load_norm(j.tstats, target_row(j, tr.r, n));
    if (resid) dn = load_norm(j.dstats, (long long)tr.r * j.gamma + n);
  }
}

// Work unit: one column tile of W2 against a pair of row blocks (2*mp, 2*mp + 1; the last pair
// of an odd count holds one block). The B tile is loaded once and feeds one MMA group per row
// block, and both blocks' A operands stay in tensor memory while the CTA works on the pair.
template <int MODE, bool ARGMAX, bool GATHER>
__global__ void __launch_bounds__(Roles<GATHER>::kThreads, 1)
    markov_tc_kernel(const __grid_constant__ CUtensorMap map_w2,
                     const __grid_constant__ CUtensorMap map_u,
                     const __grid_constant__ CUtensorMap map_t, const TcParams P) {
  using C = Cfg<MODE>;
  using RL = Roles<GATHER>;
  constexpr int BN = C::kBN;
  constexpr int KB = C::kBStages, KU = C::kUStages, KA = C::kAccStages;
  constexpr bool kPair = MODE != MODE_STATS;  // needs target tiles
  constexpr int kHalf = BN / 2;               // columns per epilogue warp

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const RowJob& j = P.j;
  const int ka_n = j.rank / 64;
  unsigned char* sB = smem;                                         // KB stages
  unsigned char* sU = sB + KB * C::kBStageBytes;                    // KU stages
  unsigned char* sT = sU + KU * C::kTileBytes;                      // KU stages (pair modes)
  unsigned char* tail = sT + (kPair ? KU * C::kTileBytes : 0);
  uint64_t* b_full = reinterpret_cast<uint64_t*>(tail);
  uint64_t* b_empty = b_full + KB;
  uint64_t* u_full = b_empty + KB;
  uint64_t* u_empty = u_full + KU;
  uint64_t* acc_full = u_empty + KU;
  uint64_t* acc_empty = acc_full + KA;
  uint64_t* a_full = acc_empty + KA;  // [2]: A of the pair's first / second row block
  uint64_t* a_empty = a_full + 2;
  uint64_t* drain = a_empty + 1;
  uint64_t* scr_free = drain + 1;  // the first A gather is done with its scratch (B stage 1)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(scr_free + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // gathered rows: T and U row indices of the pair's two row blocks, [block][row]; each copier
  // writes and reads only the entries of its own rows
  int* row_t = reinterpret_cast<int*>(tail + 256);
  // scratch of the CTA's first A gather (4 KB per epilogue warp): the second W2 stage, or with
  // a single W2 stage the second T stage; whoever fills it first waits for scr_free
  constexpr bool kScrInB = KB >= 2;
  static_assert(kScrInB ? kEpiWarps * 4096 <= C::kBStageBytes
                        : (kPair && KU >= 2 && kEpiWarps * 4096 <= C::kTileBytes),
                "gather scratch");
  unsigned char* const scr_base = kScrInB ? sB + C::kBStageBytes : sT + C::kTileBytes;
  int* row_u = row_t + 2 * kBM;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* status = j.status;

  // contiguous range of units for this CTA
  const int n_nt = P.t.n_nt;
  const int n_mp = (P.t.n_mt + 1) / 2;
  const long long total = (long long)n_mp * n_nt;
  const long long u_begin = total * blockIdx.x / gridDim.x;
  const long long u_end = total * (blockIdx.x + 1) / gridDim.x;
  const int mp_first = (int)(u_begin / n_nt), nt_first = (int)(u_begin % n_nt);
  const int n_mt = P.t.n_mt;

  if (threadIdx.x == 0) {
    for (int s = 0; s < KB; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < KU; ++s) {
      mbar_init(&u_full[s], GATHER ? 32 * RL::kCopiers : 1);  // gathered: one per copier lane
      mbar_init(&u_empty[s], kEpiWarps);
    }
    for (int s = 0; s < KA; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], kEpiWarps);
    }
    mbar_init(&a_full[0], kEpiWarps);
    mbar_init(&a_full[1], kEpiWarps);
    mbar_init(a_empty, 1);
    mbar_init(drain, 1);
    mbar_init(scr_free, kEpiWarps);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // When this launch is chained to the kernel that drew the previous tokens, the W2 and logit
  // tiles (inputs that no kernel writes) start loading before that kernel's completion; the
  // warps that read its tokens or write the partials it reads pass grid_dep_wait first.

  const bool epi_warp = warp >= RL::kFirstEpi && warp < RL::kFirstEpi + kEpiWarps;
  if (!epi_warp) {
    if constexpr (GATHER) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RL::kRegsLow));
    if (warp == 0) {
      // ---------------------------------------------------------------- W2 (B) producer
      const uint64_t pol_keep = policy_evict_last();
      int bs = 0;
      uint32_t bph = 0;
      bool ok = true;
      int nt = nt_first;
      for (long long u = u_begin; u < u_end && ok; ++u) {
        const int n0 = nt * BN;
        if (++nt == n_nt) nt = 0;
        ok = mbar_wait(&b_empty[bs], bph ^ 1, abort, status);
        if (ok && kScrInB && u == u_begin + 1) ok = mbar_wait(scr_free, 0, abort, status);
        if (ok && lane == 0 && !(P.stall && u == u_begin)) {
          mbar_arrive_expect_tx(&b_full[bs], ka_n * C::kBAtomBytes);
          for (int ka = 0; ka < ka_n; ++ka)
            tma_load_2d(sB + bs * C::kBStageBytes + ka * C::kBAtomBytes, &map_w2, ka * 64, n0,
                        &b_full[bs], pol_keep);
        }
        if (++bs == KB) { bs = 0; bph ^= 1; }
      }
      // drain: every issued copy lands before the CTA moves on
      if (lane == 0)
        for (int s = 0; s < KB; ++s) mbar_drain(&b_full[s], (s < bs) ? bph : (bph ^ 1));
    } else if (warp == 2 || (GATHER && (warp == 3 || warp >= 12))) {
      // ---------------------------------------------------------------- U / T producer
      const uint64_t pol_stream = policy_evict_first();
      int us = 0;
      uint32_t uph = 0;
      bool ok = true;
      int mp = mp_first, nt = nt_first, rows_mp = -1;
      // gathered rows: copiers 0..2 take the T rows and 3..5 the U rows of every block, each
      // the rows [r_lo, r_hi) (42, 42 and 44 of 128)
      const int cw = warp <= 3 ? warp - 2 : warp - 10;
      const bool tside = cw < 3;
      const int sub = cw % 3;
      const int r_lo = (sub * kBM / 3) & ~1, r_hi = sub == 2 ? kBM : ((sub + 1) * kBM / 3) & ~1;
      if constexpr (GATHER) grid_dep_wait();  // the final rows come from the acceptance scan
      // gathered row indices of the pair's two row blocks, loaded once per pair into a table
      // (rows past R and the U rows of bonus rows point at row 0 and are ignored)
      for (long long u = u_begin; u < u_end && ok; ++u) {
        const int n0 = nt * BN;
        const int nb = 2 * mp + 1 < n_mt ? 2 : 1;
        if constexpr (GATHER) {
          // each copier builds the table entries of its own rows in both blocks (2 x 44 at
          // most), with every load of a lane in flight at once
          if (mp != rows_mp) {
            rows_mp = mp;
            const int nr = r_hi - r_lo;
            int nn[3], kind[3];
#pragma unroll
            for (int t = 0; t < 3; ++t) {
              const int e = lane + 32 * t, sbx = e >= nr ? 1 : 0, ii = r_lo + e - sbx * nr;
              const int r = (2 * mp + sbx) * kBM + ii;
              const bool in = e < 2 * nr && sbx < nb && r < j.R;
              nn[t] = in ? j.final_n[r] : -1;
              kind[t] = in && !tside ? j.final_kind[r] : 0;
            }
#pragma unroll
            for (int t = 0; t < 3; ++t) {
              const int e = lane + 32 * t, sbx = e >= nr ? 1 : 0, ii = r_lo + e - sbx * nr;
              const int r = (2 * mp + sbx) * kBM + ii;
              if (e < 2 * nr) {
                if (tside) row_t[sbx * kBM + ii] = nn[t] >= 0 ? (int)target_row(j, r, nn[t]) : 0;
                else row_u[sbx * kBM + ii] = kind[t] ? r * j.gamma + nn[t] : 0;
              }
            }
            __syncwarp();
          }
        }
        for (int sb = 0; sb < nb && ok; ++sb) {
          const int mt = 2 * mp + sb;
          ok = mbar_wait(&u_empty[us], uph ^ 1, abort, status);
          // the first fill of T stage 1 waits until the first A gather is done with it
          if (ok && !kScrInB && us == 1 && uph == 0 && (!GATHER || tside))
            ok = mbar_wait(scr_free, 0, abort, status);
          if (!ok) break;
          unsigned char* du = sU + us * C::kTileBytes;
          unsigned char* dt = sT + us * C::kTileBytes;
          if constexpr (!GATHER) {
            if (lane == 0) {
              const TileRow tr = tile_row(j, P.t, mt, 0);
              const int r0 = tr.r, kk = tr.k - 1;
              mbar_arrive_expect_tx(&u_full[us], (kPair ? 2u : 1u) * C::kTileBytes);
              for (int b = 0; b < C::kBoxes; ++b) {
                tma_load_3d(du + b * kBoxBytes, &map_u, n0 + b * 64, kk, r0, &u_full[us],
                            pol_stream);
                if constexpr (kPair)
                  tma_load_3d(dt + b * kBoxBytes, &map_t, n0 + b * 64, kk, r0, &u_full[us],
                              pol_stream);
              }
            }
          } else {
            // final rows of rejection verification: per instruction, 8 lanes per 64-column box
            // copy one row's piece (16 bytes each) of this copier's tensor (T or U), so a warp
            // moves 4 / kBoxes whole row pieces; pieces land in the 128-byte swizzled box layout,
            // and columns past V are zero-filled without a read
            constexpr int kLanesPerRow = 8 * C::kBoxes, kRowsPerInstr = 32 / kLanesPerRow;
            static_assert(kRowsPerInstr == 2, "copier row ranges are even");
            const unsigned short* src = static_cast<const unsigned short*>(tside ? j.T : j.U);
            const int* tab = tside ? row_t : row_u;
            const uint32_t dst = smem_u32(tside ? dt : du);
            const int c = lane % kLanesPerRow;          // 16-byte chunk of the row piece
            const int bx = c >> 3, cc = c & 7;          // box and chunk within the box
            const uint32_t nb16 = n0 + 8 * c < j.V ? 16u : 0u;
#pragma unroll 4
            for (int k = 0; k < (r_hi - r_lo) / kRowsPerInstr; ++k) {
              const int i = r_lo + kRowsPerInstr * k + lane / kLanesPerRow;  // row of the block
              const long long ro = (long long)tab[sb * kBM + i] * j.V + n0 + 8 * c;
              const uint32_t so = bx * kBoxBytes + i * 128 + ((cc ^ (i & 7)) << 4);
              cp_async16(dst + so, src + (nb16 ? ro : 0), nb16, pol_stream);
            }
            cp_async_arrive(&u_full[us]);
          }
          if (++us == KU) { us = 0; uph ^= 1; }
        }
        if (++nt == n_nt) { nt = 0; ++mp; }
      }
      if (lane == 0)
        for (int s = 0; s < KU; ++s) mbar_drain(&u_full[s], (s < us) ? uph : (uph ^ 1));
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16(kBM, BN);
      if (lane == 0) {
        bool ok = true;
        int bs = 0, as = 0;
        uint32_t bph = 0;
        uint32_t accph[KA] = {};
        int mp = mp_first, nt = nt_first, cur_mp = -1, pair_i = -1;
        for (long long u = u_begin; u < u_end && ok; ++u) {
          const int nb = 2 * mp + 1 < n_mt ? 2 : 1;
          const bool first = mp != cur_mp;
          if (first) {
            cur_mp = mp;
            ++pair_i;
          }
          ok = mbar_wait(&b_full[bs], bph, abort, status);
          if (!ok) break;
          tc_fence_after();
          for (int sb = 0; sb < nb && ok; ++sb) {
            if (first) {
              ok = mbar_wait(&a_full[sb], pair_i & 1, abort, status);
              if (!ok) break;
            }
            ok = mbar_wait(&acc_empty[as], accph[as] ^ 1, abort, status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d = tmem + as * BN;
            const uint32_t a = tmem + C::kAccCols + sb * C::kACols;
            for (int ka = 0; ka < ka_n; ++ka) {
              const uint32_t b_base = smem_u32(sB + bs * C::kBStageBytes + ka * C::kBAtomBytes);
              // K = 16 per instruction: 8 tensor-memory columns of A, 32 bytes of a B row
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ta(d, a + ka * 32 + ks * 8, sw128_desc(b_base + ks * 32), idesc,
                            (ka | ks) != 0);
            }
            mma_commit(&acc_full[as]);
            accph[as] ^= 1;
            if (++as == KA) as = 0;
          }
          if (!ok) break;
          mma_commit(&b_empty[bs]);
          if (++bs == KB) { bs = 0; bph ^= 1; }
          if (++nt == n_nt) { nt = 0; ++mp; }
          if (u + 1 == u_end || mp != cur_mp) mma_commit(a_empty);  // last unit of this pair
        }
        // all MMAs issued by this thread complete before tensor memory is released
        mma_commit(drain);
        mbar_drain(drain, 0);
      }
      __syncwarp();
    }
  } else {
    if constexpr (GATHER) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(RL::kRegsHigh));
    // ---------------------------------------------------------------- epilogue
    grid_dep_wait();
    const int ew = warp - RL::kFirstEpi;
    const int q = warp & 3;          // TMEM lane quarter
    const int h = ew >> 2;           // column half
    const int i = q * 32 + lane;     // row within the tile (TMEM lane)
    int as = 0, us = 0;
    uint32_t accph[KA] = {}, uph = 0, aeph = 0;
    int mp = mp_first, nt = nt_first, cur_mp = -1;
    bool ok = true;
    // this row's normalisers in the pair's two row blocks (pair modes)
    Norm dn0 = {0.0f, 0.0f}, tn0 = {0.0f, 0.0f}, dn1 = {0.0f, 0.0f}, tn1 = {0.0f, 0.0f};
    bool rs0 = true, rs1 = true;
    for (long long u = u_begin; u < u_end && ok; ++u) {
      const int n0 = nt * BN;
      const int nb = 2 * mp + 1 < n_mt ? 2 : 1;
      if (mp != cur_mp) {
        if (cur_mp >= 0) {
          ok = mbar_wait(a_empty, aeph, abort, status);
          aeph ^= 1;
          if (!ok) break;
        }
        const bool first_pair = cur_mp < 0;
        cur_mp = mp;
        // gather A into tensor memory: thread (q, h) owns row i of each block of the pair and
        // half h of its K. The previous tokens first (a bad one is flagged and its row read as
        // zeros), then every W1 chunk in flight at once, then tcgen05.st.
        const int per = j.rank / 16;  // 16-byte chunks of a half row (<= 16)
        int src_row[2] = {-1, -1};
        for (int sb = 0; sb < nb; ++sb) {
          const TileRow tr = tile_row(j, P.t, 2 * mp + sb, i);
          if (!tr.valid) continue;
          int prev;
          if (j.map == MAP_FINAL) {
            const int n = j.final_n[tr.r];
            prev = n == 0 ? j.anchors[tr.r] : j.tokens[(size_t)tr.r * j.gamma + n - 1];
          } else {
            prev = tr.k == 1 ? j.anchors[tr.r] : j.tokens[(size_t)tr.r * j.gamma + tr.k - 2];
          }
          if (prev < 0 || prev >= j.V) atomicOr(status, SPEC_DEV_BAD_TOKEN);
          else src_row[sb] = prev;
        }
        const uint4* w1 = reinterpret_cast<const uint4*>(j.W1);
        const int row_chunks = 2 * per;  // 16-byte chunks of a W1 row
        if (first_pair) {
          // The CTA's first pair reads the rows whole (eight lanes per 128-byte piece, so an
          // instruction touches 4 lines rather than 32) and turns them into one row per lane
          // through the 4 KB per-warp scratch, which is not refilled before it is released.
          // Piece p of a half row is chunks 8p..8p+7; chunk c of warp row rl sits at slot
          // c ^ (rl & 7), so stores and loads are conflict-free.
          const uint32_t scr = smem_u32(scr_base) + ew * 4096;
          // Softmax-partial and residual passes: four lanes per piece, 32 bytes each (eight rows
          // per instruction), which halves the loads in flight; slot k of v holds the piece's
          // chunk pair of row 8(k/2) + lane/4, half k%2. TV pass: eight lanes per piece, 16 bytes
          // each (the wide loads made that pass slower); slot k holds row 4k + lane/8.
          constexpr bool kWide = MODE != MODE_TV;
          uint4 v[2][2][8];
#pragma unroll
          for (int sb = 0; sb < 2; ++sb)
#pragma unroll
            for (int p = 0; p < 2; ++p) {
              if constexpr (kWide) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int rl = 8 * k + (lane >> 2), c = 8 * p + 2 * (lane & 3);
                  const int row = __shfl_sync(0xffffffffu, src_row[sb], rl);
                  uint4 a = make_uint4(0, 0, 0, 0), b = a;
                  // per is a multiple of 4 and c even, so chunk c + 1 is in the row too
                  if (row >= 0 && c < per) {
                    const uint4* src = w1 + (size_t)row * row_chunks + h * per + c;
                    if (P.w1_32) {
                      asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                                   : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x),
                                     "=r"(b.y), "=r"(b.z), "=r"(b.w)
                                   : "l"(src));
                    } else {
                      a = __ldg(src);
                      b = __ldg(src + 1);
                    }
                  }
                  v[sb][p][2 * k] = a;
                  v[sb][p][2 * k + 1] = b;
                }
              } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const int rl = 4 * k + (lane >> 3), c = 8 * p + (lane & 7);
                  const int row = __shfl_sync(0xffffffffu, src_row[sb], rl);
                  v[sb][p][k] = make_uint4(0, 0, 0, 0);
                  if (row >= 0 && c < per)
                    v[sb][p][k] = __ldg(w1 + (size_t)row * row_chunks + h * per + c);
                }
              }
            }
#pragma unroll
          for (int sb = 0; sb < 2; ++sb) {
            if (sb >= nb) break;
            const uint32_t a_addr = tmem + ((uint32_t)(q * 32) << 16) + C::kAccCols +
                                    sb * C::kACols + h * (j.rank / 4);
#pragma unroll
            for (int p = 0; p < 2; ++p) {
              if constexpr (kWide) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int rl = 8 * k + (lane >> 2), cc = 2 * (lane & 3);
                  sts128(scr + rl * 128 + ((cc ^ (rl & 7)) << 4), v[sb][p][2 * k]);
                  sts128(scr + rl * 128 + (((cc + 1) ^ (rl & 7)) << 4), v[sb][p][2 * k + 1]);
                }
              } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const int rl = 4 * k + (lane >> 3);
                  sts128(scr + rl * 128 + (((lane & 7) ^ (rl & 7)) << 4), v[sb][p][k]);
                }
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
              // chunk c of the half holds K elements 8c..8c+7 = columns 4c..4c+3 of the half
              if (8 * p < per) tmem_st16(a_addr + 32 * p, w);
              if (8 * p + 4 < per) tmem_st16(a_addr + 32 * p + 16, w + 16);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[sb]);
          }
          // the scratch's generic-proxy accesses are ordered before the W2 copy into it
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(scr_free);
        } else {
          for (int sb = 0; sb < nb; ++sb) {
            uint32_t w[64];
#pragma unroll
            for (int it = 0; it < 16; ++it) {
              const uint4 x = (src_row[sb] >= 0 && it < per)
                                  ? __ldg(w1 + (size_t)src_row[sb] * row_chunks + h * per + it)
                                  : make_uint4(0, 0, 0, 0);
              w[4 * it] = x.x;
              w[4 * it + 1] = x.y;
              w[4 * it + 2] = x.z;
              w[4 * it + 3] = x.w;
            }
            const uint32_t a_addr = tmem + ((uint32_t)(q * 32) << 16) + C::kAccCols +
                                    sb * C::kACols + h * (j.rank / 4);
#pragma unroll
            for (int b = 0; b < 4; ++b)
              if (4 * b < per) tmem_st16(a_addr + 16 * b, w + 16 * b);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[sb]);
          }
        }
        if constexpr (kPair) {
          row_norms_tc<MODE>(j, tile_row(j, P.t, 2 * mp, i), dn0, tn0, rs0);
          if (nb > 1) row_norms_tc<MODE>(j, tile_row(j, P.t, 2 * mp + 1, i), dn1, tn1, rs1);
        }
      }
      const int col0 = h * kHalf;  // first tile column of this warp
      const bool tail = n0 + BN > j.V;
#pragma unroll 1
      for (int sb = 0; sb < nb && ok; ++sb) {
        const TileRow tr = tile_row(j, P.t, 2 * mp + sb, i);
        const bool live = tr.valid && n0 + col0 < j.V;
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + as * BN + col0;
        // allowed-token bits of this thread's columns (grammar-masked drafting), loaded before
        // the waits so that the load is in flight meanwhile
        uint32_t mlo = ~0u, mhi = ~0u;
        if (j.mask && live) {
          const uint32_t* mr = j.mask + (size_t)tr.r * j.mask_words + ((n0 + col0) >> 5);
          mlo = mr[0];
          if (kHalf == 64) mhi = n0 + col0 + 32 < j.V ? mr[1] : 0u;
        }
        ok = mbar_wait(&acc_full[as], accph[as], abort, status);
        if (!ok) break;
        tc_fence_after();
        ok = mbar_wait(&u_full[us], uph, abort, status);
        if (!ok) break;
        const size_t o = (size_t)tr.prow * P.nseg + (n0 + col0) / kHalf;
        const uint32_t u_base = smem_u32(sU + us * C::kTileBytes);
        const uint32_t t_base = smem_u32(sT + us * C::kTileBytes);
        if constexpr (MODE == MODE_STATS) {
          // TMEM reads and shared-memory reads first, then release the stages
          uint32_t braw[kHalf];
          tmem_ld32_async(taddr, braw);
          if constexpr (kHalf == 64) tmem_ld32_async(taddr + 32, braw + 32);
          uint4 uw[kHalf / 8];
#pragma unroll
          for (int c = 0; c < kHalf / 8; ++c) {
            const int col = col0 + 8 * c;
            const int b = col >> 6, cc = (col & 63) >> 3;
            uw[c] = lds128(u_base + b * kBoxBytes + i * 128 + ((cc ^ (i & 7)) << 4));
          }
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&acc_empty[as]);
            mbar_arrive(&u_empty[us]);
          }
          float m, sum;
          int idx;
          stats_partial64<ARGMAX>(braw, uw, j.scale, n0 + col0, j.V, tail, j.mask != nullptr, mlo,
                                  mhi, m, sum, idx);
          if (live) {
            P.pm[o] = m;
            P.ps[o] = sum;
            if (ARGMAX) P.pi[o] = idx;
          }
        } else {
          const Norm dn = sb ? dn1 : dn0, tn = sb ? tn1 : tn0;
          const bool resid = sb ? rs1 : rs0;
          // 32 columns at a time (one rolled loop, so the code stays small): their accumulators
          // and logits, then their terms; the stages are released after the last reads.
          // Branch-free: every column's two probabilities are computed, then selected, so that
          // the exponentials of all columns overlap; four partial sums, in column order.
          float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          const bool masked = j.mask != nullptr;
#pragma unroll 1
          for (int hh = 0; hh < kHalf / 32; ++hh) {
            uint32_t braw[32];
            tmem_ld32_async(taddr + 32 * hh, braw);
            uint4 uw[4], tw[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int col = col0 + 32 * hh + 8 * c;
              const int b = col >> 6, cc = (col & 63) >> 3;
              const uint32_t off = b * kBoxBytes + i * 128 + ((cc ^ (i & 7)) << 4);
              uw[c] = lds128(u_base + off);
              tw[c] = lds128(t_base + off);
            }
            tmem_wait_ld();
            if (hh == kHalf / 32 - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                mbar_arrive(&acc_empty[as]);
                mbar_arrive(&u_empty[us]);
              }
            }
            if (!live) continue;
            const int vb = n0 + col0 + 32 * hh;   // first column of these 32
            const uint32_t mbits = hh ? mhi : mlo;  // their allowed-token bits
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float uv[8], tv[8];
              unpack_bf16x8(tw[c], tv);
              unpack_bf16x8(uw[c], uv);
              // Outside the element loop, in the tiles that have them: a column past V gets both
              // logits -inf (its term is 0 in both modes, even beside a non-finite normaliser)
              // and a disallowed token the base logit -inf (p_d = 0).
              if (tail) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  if (vb + c * 8 + e >= j.V) tv[e] = uv[e] = -INFINITY;
              }
              if (masked) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  if (!((mbits >> (c * 8 + e)) & 1u)) uv[e] = -INFINITY;
              }
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                float x;
                if constexpr (MODE == MODE_TV) {
                  // min(p_t, p_d) = 2^min(a_t, a_d) for the exponents a of prob_of: exp is
                  // increasing, so one exponential per element instead of two
                  const float at = ((tv[e] * j.scale - tn.m) - tn.lz) * kLog2e;
                  const float ad =
                      (((uv[e] + __uint_as_float(braw[c * 8 + e])) * j.scale - dn.m) - dn.lz) *
                      kLog2e;
                  x = fast_exp2(fminf(at, ad));
                } else {
                  const float pt = prob_of(tv[e] * j.scale, tn);
                  const float pd =
                      prob_of((uv[e] + __uint_as_float(braw[c * 8 + e])) * j.scale, dn);
                  x = fmaxf(pt - (resid ? pd : 0.0f), 0.0f);  // bonus rows: p_t
                }
                acc[e & 3] += x;
              }
            }
          }
          if (live) P.ps[o] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        }
        if (++us == KU) { us = 0; uph ^= 1; }
        accph[as] ^= 1;
        if (++as == KA) as = 0;
      }
      if (++nt == n_nt) { nt = 0; ++mp; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  if (!encode_fn()) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                     strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
constexpr size_t smem_bytes() {
  using C = Cfg<MODE>;
  return 1024 + C::kBStages * C::kBStageBytes +
         (MODE != MODE_STATS ? 2 : 1) * C::kUStages * C::kTileBytes + 512 +
         (MODE != MODE_STATS ? 4 * kBM * 4 : 0);  // gathered row table (pair modes)
}

// the largest dynamic shared memory a CTA may opt into (227 KB)
static_assert(smem_bytes<MODE_STATS>() <= 232448 && smem_bytes<MODE_TV>() <= 232448 &&
                  smem_bytes<MODE_RESID>() <= 232448,
              "shared-memory budget");

template <int MODE, bool ARGMAX, bool GATHER>
cudaError_t launch_t(const TcParams& p, const CUtensorMap& w2, const CUtensorMap& u,
                     const CUtensorMap& t, int grid, cudaStream_t s) {
  const size_t smem = smem_bytes<MODE>();
  auto k = markov_tc_kernel<MODE, ARGMAX, GATHER>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(k, dim3(grid), dim3(Roles<GATHER>::kThreads), smem, s, p.j.pdl != 0, w2,
                       u, t, p);
}

}  // namespace tc

int markov_tc_seg(int mode) {
  return mode == MODE_STATS ? tc::Cfg<MODE_STATS>::kSeg
                            : (mode == MODE_TV ? tc::Cfg<MODE_TV>::kSeg : tc::Cfg<MODE_RESID>::kSeg);
}

bool markov_tc_supported(int udt, int wdt, int rank, int V, const void* U, const void* T,
                         const void* W1, const void* W2) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (udt != SPEC_BF16 || wdt != SPEC_BF16) return false;
  if (rank <= 0 || rank > 256 || rank % 64 != 0 || V % 8 != 0) return false;
  if (!al(U) || !al(T) || !al(W1) || !al(W2)) return false;
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return false;
  if (major < 10) return false;
  return tc::encode_fn() != nullptr;
}

int g_stall_next = 0;  // spec_test_stall_next_markov

int take_stall_request() { return __atomic_exchange_n(&g_stall_next, 0, __ATOMIC_RELAXED); }

bool make_tensor_map_bf16(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                          const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  return tc::make_map(m, base, rank, dims, strides_bytes, box);
}

cudaError_t launch_markov_tc(const RowJob& j, float* pm, float* ps, int* pi, bool argmax,
                             cudaStream_t s) {
  using namespace tc;
  TraceScope ts(SPEC_KCLASS_MARKOV, s);
  const bool pair = j.mode != MODE_STATS;
  const int BN = j.mode == MODE_STATS ? Cfg<MODE_STATS>::kBN
                 : (j.mode == MODE_TV ? Cfg<MODE_TV>::kBN : Cfg<MODE_RESID>::kBN);
  TcParams p;
  p.j = j;
  p.pm = pm;
  p.ps = ps;
  p.pi = pi;
  const int rb = (j.R + kBM - 1) / kBM;
  p.t.rb = rb;
  p.t.n_mt = j.map == MAP_ALL_POS ? rb * j.gamma : rb;
  p.t.n_nt = (j.V + BN - 1) / BN;
  p.nseg = (j.V + BN / 2 - 1) / (BN / 2);
  p.stall = take_stall_request();
  p.w1_32 = (reinterpret_cast<uintptr_t>(j.W1) & 31) == 0;
  // work units: one column tile against a pair of row blocks
  const long long total = (long long)((p.t.n_mt + 1) / 2) * p.t.n_nt;
  if (total == 0) return cudaSuccess;
  const int grid = (int)(total < num_sms() ? total : num_sms());

  CUtensorMap w2, u, t;
  memset(&u, 0, sizeof u);
  memset(&t, 0, sizeof t);
  {
    const cuuint64_t dims[2] = {(cuuint64_t)j.rank, (cuuint64_t)j.V};
    const cuuint64_t str[1] = {(cuuint64_t)j.rank * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)BN};
    if (!make_map(&w2, j.W2, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  const bool gather = j.map == MAP_FINAL;
  if (!gather) {
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kBM};
    const cuuint64_t du[3] = {(cuuint64_t)j.V, (cuuint64_t)j.gamma, (cuuint64_t)j.R};
    const cuuint64_t su[2] = {(cuuint64_t)j.V * 2, (cuuint64_t)j.V * 2 * j.gamma};
    if (!make_map(&u, j.U, 3, du, su, box)) return cudaErrorInvalidValue;
    if (pair) {
      const cuuint64_t dt[3] = {(cuuint64_t)j.V, (cuuint64_t)j.gamma + 1, (cuuint64_t)j.R};
      const cuuint64_t st[2] = {(cuuint64_t)j.V * 2, (cuuint64_t)j.V * 2 * (j.gamma + 1)};
      if (!make_map(&t, j.T, 3, dt, st, box)) return cudaErrorInvalidValue;
    }
  }  // gathered rows are copied with cp.async: their maps stay zero and unused
  if (j.mode == MODE_STATS) {
    if (argmax) return launch_t<MODE_STATS, true, false>(p, w2, u, t, grid, s);
    return launch_t<MODE_STATS, false, false>(p, w2, u, t, grid, s);
  }
  if (j.mode == MODE_TV) return launch_t<MODE_TV, false, false>(p, w2, u, t, grid, s);
  return launch_t<MODE_RESID, false, true>(p, w2, u, t, grid, s);
}

}  // namespace spec

extern "C" int spec_test_stall_next_markov(void) {
  __atomic_store_n(&spec::g_stall_next, 1, __ATOMIC_RELAXED);
  return SPEC_OK;
}
