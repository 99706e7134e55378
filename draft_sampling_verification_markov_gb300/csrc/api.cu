// api.cu -- the extern "C" entry points of libspecmarkov: host-side validation, workspace
// carving and the sequence of passes each operation enqueues on the caller's stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "spec_markov.h"

namespace spec {

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  static int cached[64] = {0};
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

namespace {

struct TraceState {
  cudaEvent_t* begin = nullptr;
  cudaEvent_t* end = nullptr;
  int capacity = 0;
  int count = 0;
  int open = -1;  // index of the launch whose end event is pending
};
TraceState g_trace[SPEC_KCLASS_COUNT];
unsigned long long g_launches = 0;

}  // namespace

// Inside a stream capture a record must be external to stay a timing record of the graph;
// outside a capture the external flag is not accepted.
static void record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

void trace_begin(int kclass, cudaStream_t s) {
  __atomic_fetch_add(&g_launches, 1ull, __ATOMIC_RELAXED);
  TraceState& t = g_trace[kclass];
  if (t.count < t.capacity) {
    record(t.begin[t.count], s);
    t.open = t.count;
  }
}

void trace_end(int kclass, cudaStream_t s) {
  TraceState& t = g_trace[kclass];
  if (t.open >= 0) {
    record(t.end[t.open], s);
    t.open = -1;
    ++t.count;
  }
}

bool trace_active() {
  for (const TraceState& t : g_trace)
    if (t.capacity > 0) return true;
  return false;
}

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kHeader = 256;                        // status word + spare
constexpr size_t kFixed = kSyncOffset + kSyncBytes;    // header + persistent-proposal counters
static_assert(kSyncOffset >= kHeader, "counters after the header");

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

int markov_nseg(int V) { return cdiv(V, kMarkovMinSeg); }
int stream_nseg(int V) { return cdiv(V, kStreamSeg); }

struct Layout {
  size_t pm, ps, pi;  // partial arrays, `entries` elements each
  size_t tstats, dstats, final_n, final_kind;
  size_t total;
  size_t entries;
};

// Partial entries (rows x segments) of the largest pass of an op.
size_t partial_entries(int op, int R, int gamma, int V, int rank) {
  const size_t tr = (size_t)R * (gamma + 1), dr = (size_t)R * gamma;
  const size_t seg_draft = rank > 0 ? markov_nseg(V) : stream_nseg(V);
  const size_t tgt = tr * stream_nseg(V);
  size_t e = 0;
  switch (op) {
    case SPEC_OP_PROPOSE:
      e = (size_t)R * (rank > 0 ? 1 : gamma) * seg_draft;
      // the persistent proposal: 64-column partials, then 2 coarse ones per tile range
      if (rank > 0) {
        const size_t pe = (size_t)R * (cdiv(V, 64) + 2 * kMaxPropGrid);
        e = e > pe ? e : pe;
      }
      break;
    case SPEC_OP_VERIFY_GREEDY: e = tr; break;
    case SPEC_OP_MTP_GREEDY: {
      // one partial per streamed item, or the two-call form's proposal and verification
      const size_t fe = (size_t)R * (2 * (size_t)gamma + 1) * cdiv(V, kMtpChunk);
      const size_t pe = dr * stream_nseg(V);
      e = fe > pe ? fe : pe;
      e = e > tr ? e : tr;
      break;
    }
    case SPEC_OP_TARGET_STATS: e = tgt; break;
    case SPEC_OP_VERIFY_REJECTION: e = tgt > (size_t)R * seg_draft ? tgt : (size_t)R * seg_draft; break;
    case SPEC_OP_TV_CONFIDENCE: e = tgt > dr * seg_draft ? tgt : dr * seg_draft; break;
    default: e = 0; break;
  }
  return e;
}

Layout layout(int op, int R, int gamma, int V, int rank) {
  Layout L;
  size_t e = 0;
  if (op == SPEC_OP_ALL) {
    for (int o = 0; o < SPEC_OP_ALL; ++o) {
      const size_t x = partial_entries(o, R, gamma, V, rank);
      e = x > e ? x : e;
    }
  } else {
    e = partial_entries(op, R, gamma, V, rank);
  }
  L.entries = e;
  size_t off = kFixed;
  L.pm = off; off = align_up(off + e * sizeof(float));
  L.ps = off; off = align_up(off + e * sizeof(float));
  L.pi = off; off = align_up(off + e * sizeof(int));
  L.tstats = off; off = align_up(off + (size_t)R * (gamma + 1) * 2 * sizeof(float));
  L.dstats = off; off = align_up(off + (size_t)R * gamma * 2 * sizeof(float));
  L.final_n = off; off = align_up(off + (size_t)R * sizeof(int32_t));
  L.final_kind = off; off = align_up(off + (size_t)R * sizeof(int32_t));
  L.total = off;
  return L;
}

struct Ws {
  uint32_t* status;
  float* pm;
  float* ps;
  int* pi;
  float* tstats;
  float* dstats;
  int32_t* final_n;
  int32_t* final_kind;
};

Ws carve(void* ws, const Layout& L) {
  char* b = static_cast<char*>(ws);
  return Ws{reinterpret_cast<uint32_t*>(b), reinterpret_cast<float*>(b + L.pm),
            reinterpret_cast<float*>(b + L.ps), reinterpret_cast<int*>(b + L.pi),
            reinterpret_cast<float*>(b + L.tstats), reinterpret_cast<float*>(b + L.dstats),
            reinterpret_cast<int32_t*>(b + L.final_n), reinterpret_cast<int32_t*>(b + L.final_kind)};
}

bool dtype_ok(int d) { return d == SPEC_F32 || d == SPEC_BF16; }
size_t esize(int d) { return d == SPEC_BF16 ? 2 : 4; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_ws(void* ws, size_t ws_bytes, int op, int R, int gamma, int V, int rank, Layout* L) {
  *L = layout(op, R, gamma, V, rank);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return SPEC_ERR_INVALID_ARG;
  if (ws_bytes < L->total) return SPEC_ERR_WORKSPACE_TOO_SMALL;
  return SPEC_OK;
}

int sizes_ok(int R, int gamma, int V) {
  if (R < 0 || gamma < 0 || V < 1) return 0;
  if ((long long)R * (gamma + 1) > (1LL << 30)) return 0;
  if ((long long)R * (gamma + 1) * V > (1LL << 46)) return 0;
  return 1;
}

int finish() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int grid_for(long long units, int per_block) {
  const long long blocks = (units + per_block - 1) / per_block;
  const long long cap = (long long)num_sms() * 8;
  return (int)(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
}

// Rows of a Markov (rank > 0) pass: tcgen05 producer when the shape allows, else CUDA cores.
// Reports the segment width of the partials it wrote.
int markov_pass(const RowJob& j, int udt, int wdt, const Ws& w, bool argmax, cudaStream_t s,
                int* seg, int* nseg) {
  if (markov_tc_supported(udt, wdt, j.rank, j.V, j.U, j.T, j.W1, j.W2)) {
    *seg = markov_tc_seg(j.mode);
    *nseg = cdiv(j.V, *seg);
    if (launch_markov_tc(j, w.pm, w.ps, w.pi, argmax, s) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
  }
  *seg = kMarkovSeg;
  *nseg = cdiv(j.V, kMarkovSeg);
  launch_ffma_partials(j, udt, wdt, *nseg, argmax, w.pm, w.ps, w.pi,
                       grid_for((long long)j.rows * *nseg, 8), s);
  return SPEC_OK;
}

bool vec_ok(const void* a, const void* b, int dtype, int V) {
  return aligned16(a) && (b == nullptr || aligned16(b)) && ((size_t)V * esize(dtype)) % 16 == 0;
}

// Target row stats (m, log Z) of all R*(gamma+1) rows into `out` (rows beyond `lengths`, or
// past toff[R] in the flattened layout, skipped).
void target_stats_pass(const void* target, int dtype, float scale, int R, int gamma, int V,
                       const int32_t* lengths, float* out, const Ws& w, cudaStream_t s,
                       const int32_t* toff = nullptr) {
  RowJob j;
  memset(&j, 0, sizeof j);
  j.rows = R * (gamma + 1);
  j.map = MAP_TARGET;
  j.mode = MODE_STATS;
  j.R = R;
  j.gamma = gamma;
  j.V = V;
  j.scale = scale;
  j.T = target;
  j.lengths = lengths;
  j.toff = toff;
  j.status = w.status;
  launch_row_stats(j, dtype, vec_ok(target, nullptr, dtype, V), out, nullptr, s);
}

}  // namespace
}  // namespace spec

using namespace spec;

extern "C" {

int spec_abi_version(void) { return SPEC_ABI_VERSION; }

unsigned long long spec_launch_count(void) { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

int spec_trace_events(int kclass, void* const* begin_events, void* const* end_events,
                      int capacity) {
  if (kclass < 0 || kclass >= SPEC_KCLASS_COUNT || capacity < 0) return SPEC_ERR_INVALID_ARG;
  if (capacity > 0 && (!begin_events || !end_events)) return SPEC_ERR_INVALID_ARG;
  TraceState& t = g_trace[kclass];
  t.begin = capacity ? reinterpret_cast<cudaEvent_t*>(const_cast<void**>(begin_events)) : nullptr;
  t.end = capacity ? reinterpret_cast<cudaEvent_t*>(const_cast<void**>(end_events)) : nullptr;
  t.capacity = capacity;
  t.count = 0;
  t.open = -1;
  return SPEC_OK;
}

int spec_trace_count(int kclass) {
  if (kclass < 0 || kclass >= SPEC_KCLASS_COUNT) return SPEC_ERR_INVALID_ARG;
  return g_trace[kclass].count;
}

const char* spec_status_string(int status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case SPEC_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SPEC_ERR_CUDA: return "CUDA error";
    case SPEC_ERR_UNSUPPORTED: return "unsupported combination";
    case SPEC_ERR_TOO_LARGE: return "size beyond the fixed scratch of this entry point";
    default: return "unknown status";
  }
}

size_t spec_workspace_bytes(int op, int R, int gamma, int V, int rank) {
  if (op < 0 || op > SPEC_OP_ALL || !sizes_ok(R, gamma, V) || rank < 0) return 0;
  return layout(op, R, gamma, V, rank).total;
}

int spec_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < kHeader || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0)
    return SPEC_ERR_INVALID_ARG;
  const size_t n = ws_bytes < kFixed ? ws_bytes : kFixed;
  if (cudaMemsetAsync(ws, 0, n, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

int spec_device_status(void* ws, size_t ws_bytes, void* stream, uint32_t* status_host, int clear) {
  if (!ws || !status_host || ws_bytes < kHeader) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_CUDA;
  *status_host = v;
  if (clear && cudaMemsetAsync(ws, 0, sizeof v, s) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

// The target normalisers of the fused proposal entry point when the proposal did not run as
// one persistent launch: a streaming pass of their own after it.
static int target_after(const void* target, float* target_stats, int dtype, float temperature,
                        int R, int gamma, int V, const Ws& w, cudaStream_t s) {
  if (target)
    target_stats_pass(target, dtype, 1.0f / temperature, R, gamma, V, nullptr, target_stats, w, s);
  return finish();
}

static int markov_propose_impl(const void* U, int u_dtype, const void* W1, const void* W2,
                               int w_dtype, int rank, const int32_t* anchors, const float* u_draft,
                               float temperature, int R, int gamma, int V, int32_t* draft_tokens,
                               float* draft_logp, float* draft_stats, void* ws, size_t ws_bytes,
                               void* stream, const uint32_t* mask, const void* target = nullptr,
                               float* target_stats = nullptr) {
  if (!sizes_ok(R, gamma, V) || rank < 0 || rank > 1024) return SPEC_ERR_INVALID_ARG;
  if (!dtype_ok(u_dtype) || (rank > 0 && !dtype_ok(w_dtype))) return SPEC_ERR_UNSUPPORTED_DTYPE;
  if (!(temperature >= 0.0f) || !isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
  Layout L;
  int rc = check_ws(ws, ws_bytes, SPEC_OP_PROPOSE, R, gamma, V, rank, &L);
  if (rc != SPEC_OK) return rc;
  if (target && (!target_stats || !(temperature > 0.0f))) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Ws w = carve(ws, L);
  if (R == 0) return SPEC_OK;
  if (gamma == 0)  // nothing to propose; the window is the bonus row alone
    return target_after(target, target_stats, u_dtype, temperature, R, gamma, V, w, s);
  if (!U || !draft_tokens) return SPEC_ERR_INVALID_ARG;
  if (rank > 0 && (!W1 || !W2 || !anchors)) return SPEC_ERR_INVALID_ARG;
  const bool greedy = u_draft == nullptr || temperature == 0.0f;

  RowJob j;
  memset(&j, 0, sizeof j);
  j.rows = R;
  j.map = MAP_POSITION;
  j.mode = MODE_STATS;
  j.R = R;
  j.gamma = gamma;
  j.V = V;
  j.scale = greedy ? 1.0f : 1.0f / temperature;
  j.U = U;
  j.W1 = W1;
  j.W2 = W2;
  j.rank = rank;
  j.anchors = anchors;
  j.tokens = draft_tokens;
  j.status = w.status;
  j.mask = mask;
  j.mask_words = (V + 31) / 32;

  SelectOut o;
  memset(&o, 0, sizeof o);
  o.kind = 0;
  o.tokens = draft_tokens;
  o.logp = draft_logp;
  o.stats = draft_stats;
  o.uni = u_draft;
  o.uni_stride = gamma;
  o.greedy = greedy;
  const int wdt = rank > 0 ? w_dtype : u_dtype;
  const bool vec = vec_ok(U, nullptr, u_dtype, V);
  if (rank == 0) {
    // no Markov head: the positions do not depend on one another, so one streaming pass and
    // one select cover all R * gamma rows (row m = r * gamma + k - 1, uniform u_draft[m])
    j.rows = R * gamma;
    j.map = MAP_ALL_POS;
    o.uni_stride = 1;
    o.uni_offset = 0;
    const int nseg = stream_nseg(V);
    launch_stream_partials(j, u_dtype, kStreamSeg, nseg, vec, true, greedy, w.pm, w.ps, w.pi,
                           grid_for((long long)j.rows * nseg, 1), s);
    j.pdl = 1;
    launch_select(j, u_dtype, wdt, kStreamSeg, nseg, w.pm, w.ps, greedy ? w.pi : nullptr, o, s);
    return target_after(target, target_stats, u_dtype, temperature, R, gamma, V, w, s);
  }
  // bf16 weights on the tensor cores: every position, selects included, in one persistent
  // launch that pipelines the positions of different request groups
  if (markov_propose_tc_supported(u_dtype, wdt, rank, R, gamma, V, U, W1, W2)) {
    o.w1 = aligned16(W1) && (rank * (int)esize(wdt)) % 16 == 0 ? W1 : nullptr;
    o.w1_row_bytes = rank * (int)esize(wdt);
    uint32_t* sync = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + kSyncOffset);
    // The target rows ride along only while the proposal's serial chain leaves SMs idle: with
    // at most two 128-request groups. With more groups the streaming CTAs are busy and the
    // normalisers are cheaper as a pass of their own.
    const bool along = target && R <= 256;
    if (launch_markov_propose_tc(j, o, w.pm, w.ps, greedy ? w.pi : nullptr, greedy, sync, s,
                                 along ? target : nullptr, target_stats,
                                 1.0f / temperature) != cudaSuccess)
      return SPEC_ERR_CUDA;
    if (target && !along) return target_after(target, target_stats, u_dtype, temperature, R, gamma, V, w, s);
    return finish();
  }
  // every launch after the first is chained to the one before it
  for (int k = 1; k <= gamma; ++k) {
    j.k = k;
    j.pdl = k > 1;
    o.uni_offset = k - 1;
    int seg, nseg;
    if (rank == 0) {
      seg = kStreamSeg;
      nseg = stream_nseg(V);
      launch_stream_partials(j, u_dtype, seg, nseg, vec, true, greedy, w.pm, w.ps, w.pi,
                             grid_for((long long)R * nseg, 1), s);
    } else {
      rc = markov_pass(j, u_dtype, wdt, w, greedy, s, &seg, &nseg);
      if (rc != SPEC_OK) return rc;
    }
    // the W1 row of each drawn token, which the next position gathers, is pulled into L2
    const int w1_row = rank * (int)esize(wdt);
    o.w1 = rank > 0 && k < gamma && aligned16(W1) && w1_row % 16 == 0 ? W1 : nullptr;
    o.w1_row_bytes = w1_row;
    j.pdl = 1;
    launch_select(j, u_dtype, wdt, seg, nseg, w.pm, w.ps, greedy ? w.pi : nullptr, o, s);
  }
  return target_after(target, target_stats, u_dtype, temperature, R, gamma, V, w, s);
}

static int verify_greedy_impl(const void* target, int t_dtype, const int32_t* draft_tokens,
                              const int32_t* lengths, const int32_t* toff, int R, int gamma,
                              int V, int32_t* accept_len, int32_t* out_tokens,
                              int32_t* next_anchor, void* ws, size_t ws_bytes, void* stream) {
  if (!sizes_ok(R, gamma, V)) return SPEC_ERR_INVALID_ARG;
  if (!dtype_ok(t_dtype)) return SPEC_ERR_UNSUPPORTED_DTYPE;
  Layout L;
  int rc = check_ws(ws, ws_bytes, SPEC_OP_VERIFY_GREEDY, R, gamma, V, 0, &L);
  if (rc != SPEC_OK) return rc;
  if (R == 0) return SPEC_OK;
  if (!target || !accept_len || (gamma > 0 && !draft_tokens)) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Ws w = carve(ws, L);
  RowJob j;
  memset(&j, 0, sizeof j);
  j.rows = R * (gamma + 1);
  j.map = MAP_TARGET;
  j.mode = MODE_STATS;
  j.R = R;
  j.gamma = gamma;
  j.V = V;
  j.scale = 1.0f;
  j.T = target;
  j.lengths = lengths;
  j.toff = toff;
  j.status = w.status;
  launch_row_stats(j, t_dtype, vec_ok(target, nullptr, t_dtype, V), nullptr, w.pi, s);
  launch_greedy_scan(R, gamma, w.pi, draft_tokens, lengths, toff, accept_len, out_tokens,
                     next_anchor, w.status, s);
  return finish();
}

int spec_verify_greedy(const void* target, int t_dtype, const int32_t* draft_tokens,
                       const int32_t* lengths, int R, int gamma, int V, int32_t* accept_len,
                       int32_t* out_tokens, int32_t* next_anchor, void* ws, size_t ws_bytes,
                       void* stream) {
  return verify_greedy_impl(target, t_dtype, draft_tokens, lengths, nullptr, R, gamma, V,
                            accept_len, out_tokens, next_anchor, ws, ws_bytes, stream);
}

int spec_verify_greedy_flat(const void* target, int t_dtype, const int32_t* draft_tokens,
                            const int32_t* lengths, const int32_t* offsets, int R, int gamma,
                            int V, int32_t* accept_len, int32_t* out_tokens,
                            int32_t* next_anchor, void* ws, size_t ws_bytes, void* stream) {
  if (R > 0 && (!lengths || !offsets)) return SPEC_ERR_INVALID_ARG;
  return verify_greedy_impl(target, t_dtype, draft_tokens, lengths, offsets, R, gamma, V,
                            accept_len, out_tokens, next_anchor, ws, ws_bytes, stream);
}

int spec_flat_layout(const int32_t* lengths, int R, int gamma, int32_t* offsets,
                     int32_t* row_req, int32_t* row_pos, void* ws, size_t ws_bytes,
                     void* stream) {
  if (R < 0 || gamma < 0 || (long long)R * (gamma + 1) > (1LL << 30)) return SPEC_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kHeader || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0)
    return SPEC_ERR_INVALID_ARG;
  if (!offsets || (R > 0 && !lengths)) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  TraceScope ts(SPEC_KCLASS_OTHER, s);
  launch_flat_layout(lengths, R, gamma, offsets, row_req, row_pos, static_cast<uint32_t*>(ws), s);
  return finish();
}

int spec_flat_pack(const void* src, int row_bytes, const int32_t* lengths,
                   const int32_t* offsets, int R, int gamma, void* dst, void* ws, size_t ws_bytes,
                   void* stream) {
  if (R < 0 || gamma < 0 || (long long)R * (gamma + 1) > (1LL << 30)) return SPEC_ERR_INVALID_ARG;
  if (row_bytes < 4 || row_bytes % 4 != 0) return SPEC_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kHeader || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0)
    return SPEC_ERR_INVALID_ARG;
  if (R == 0) return SPEC_OK;
  if (!src || !dst || !lengths || !offsets) return SPEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 3) != 0 || (reinterpret_cast<uintptr_t>(dst) & 3) != 0)
    return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  TraceScope ts(SPEC_KCLASS_OTHER, s);
  launch_flat_pack(src, row_bytes, lengths, offsets, R, gamma, dst, static_cast<uint32_t*>(ws), s);
  return finish();
}

int spec_target_stats_flat(const void* target, int t_dtype, float temperature, int R, int gamma,
                           int V, const int32_t* offsets, float* stats, void* ws,
                           size_t ws_bytes, void* stream) {
  if (!sizes_ok(R, gamma, V)) return SPEC_ERR_INVALID_ARG;
  if (!dtype_ok(t_dtype)) return SPEC_ERR_UNSUPPORTED_DTYPE;
  if (!(temperature > 0.0f) || !isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
  Layout L;
  int rc = check_ws(ws, ws_bytes, SPEC_OP_TARGET_STATS, R, gamma, V, 0, &L);
  if (rc != SPEC_OK) return rc;
  if (R == 0) return SPEC_OK;
  if (!target || !stats || !offsets) return SPEC_ERR_INVALID_ARG;
  const Ws w = carve(ws, L);
  target_stats_pass(target, t_dtype, 1.0f / temperature, R, gamma, V, nullptr, stats, w,
                    static_cast<cudaStream_t>(stream), offsets);
  return finish();
}

int spec_target_stats(const void* target, int t_dtype, float temperature, int rows, int V,
                      float* stats, void* ws, size_t ws_bytes, void* stream) {
  if (rows < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (!dtype_ok(t_dtype)) return SPEC_ERR_UNSUPPORTED_DTYPE;
  if (!(temperature > 0.0f) || !isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
  // rows are treated as one request with rows-1 proposed positions
  Layout L;
  int rc = check_ws(ws, ws_bytes, SPEC_OP_TARGET_STATS, rows > 0 ? 1 : 0, rows > 0 ? rows - 1 : 0,
                    V, 0, &L);
  if (rc != SPEC_OK) return rc;
  if (rows == 0) return SPEC_OK;
  if (!target || !stats) return SPEC_ERR_INVALID_ARG;
  const Ws w = carve(ws, L);
  target_stats_pass(target, t_dtype, 1.0f / temperature, 1, rows - 1, V, nullptr, stats, w,
                    static_cast<cudaStream_t>(stream));
  return finish();
}

static int verify_rejection_impl(const void* target, const void* U, int l_dtype, const void* W1,
                                 const void* W2, int w_dtype, int rank, const int32_t* anchors,
                                 const int32_t* draft_tokens, const float* draft_logp,
                                 const float* draft_stats, const float* target_stats,
                                 const float* u_accept, const float* u_resid, float temperature,
                                 const int32_t* lengths, int R, int gamma, int V,
                                 int32_t* accept_len, int32_t* out_tokens, int32_t* next_anchor,
                                 void* ws, size_t ws_bytes, void* stream, const uint32_t* mask,
                                 const int32_t* toff = nullptr) {
  if (!sizes_ok(R, gamma, V) || rank < 0 || rank > 1024) return SPEC_ERR_INVALID_ARG;
  if (!dtype_ok(l_dtype) || (rank > 0 && !dtype_ok(w_dtype))) return SPEC_ERR_UNSUPPORTED_DTYPE;
  if (!(temperature > 0.0f) || !isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
  Layout L;
  int rc = check_ws(ws, ws_bytes, SPEC_OP_VERIFY_REJECTION, R, gamma, V, rank, &L);
  if (rc != SPEC_OK) return rc;
  if (R == 0) return SPEC_OK;
  // without draft positions the draft side (U and the draft arrays) is never read
  if (!target || (gamma > 0 && !U) || !u_resid || !accept_len || !out_tokens)
    return SPEC_ERR_INVALID_ARG;
  if (gamma > 0 && (!draft_tokens || !draft_logp || !draft_stats || !u_accept))
    return SPEC_ERR_INVALID_ARG;
  if (rank > 0 && (!W1 || !W2 || !anchors)) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Ws w = carve(ws, L);
  const float scale = 1.0f / temperature;

  const float* tstats = target_stats;
  if (!tstats) {
    target_stats_pass(target, l_dtype, scale, R, gamma, V, lengths, w.tstats, w, s, toff);
    tstats = w.tstats;
  }
  const int w1_row = rank * (int)esize(w_dtype);
  const RowPrefetch pf = {rank > 0 && aligned16(W1) && w1_row % 16 == 0 ? W1 : nullptr, w1_row,
                          anchors};
  // chained to the target normaliser pass when this call ran it
  launch_accept(l_dtype, R, gamma, V, scale, target, tstats, draft_tokens, draft_logp, u_accept,
                lengths, toff, w.final_n, w.final_kind, accept_len, out_tokens, w.status, pf,
                tstats == w.tstats, s);

  RowJob j;
  memset(&j, 0, sizeof j);
  j.rows = R;
  j.map = MAP_FINAL;
  j.mode = MODE_RESID;
  j.R = R;
  j.gamma = gamma;
  j.V = V;
  j.scale = scale;
  j.U = U;
  j.W1 = W1;
  j.W2 = W2;
  j.rank = rank;
  j.anchors = anchors;
  j.tokens = draft_tokens;
  j.dstats = draft_stats;
  j.T = target;
  j.tstats = tstats;
  j.lengths = lengths;
  j.final_n = w.final_n;
  j.final_kind = w.final_kind;
  j.status = w.status;
  j.mask = mask;
  j.mask_words = (V + 31) / 32;
  j.toff = toff;
  j.pdl = 1;  // after the acceptance scan
  const int wdt = rank > 0 ? w_dtype : l_dtype;
  int seg, nseg;
  if (rank == 0 || gamma == 0) {
    // no Markov head, or no draft positions (every final row is a bonus row drawn from p_t
    // alone, so the draft side is never read): the streaming pass
    seg = kStreamSeg;
    nseg = stream_nseg(V);
    launch_stream_partials(j, l_dtype, seg, nseg, vec_ok(target, U, l_dtype, V), true, false,
                           w.pm, w.ps, w.pi, grid_for((long long)R * nseg, 1), s);
  } else {
    rc = markov_pass(j, l_dtype, wdt, w, false, s, &seg, &nseg);
    if (rc != SPEC_OK) return rc;
  }
  SelectOut o;
  memset(&o, 0, sizeof o);
  o.kind = 1;
  o.tokens = out_tokens;
  o.next_anchor = next_anchor;
  o.uni = u_resid;
  o.uni_stride = 1;
  o.uni_offset = 0;
  // a decoding loop proposes next from the emitted tokens: have L2 fetch their W1 rows
  o.w1 = rank > 0 && aligned16(W1) && (rank * esize(wdt)) % 16 == 0 ? W1 : nullptr;
  o.w1_row_bytes = rank * (int)esize(wdt);
  launch_select(j, l_dtype, wdt, seg, nseg, w.pm, w.ps, nullptr, o, s);
  return finish();
}

static int tv_confidence_impl(const void* U, const void* target, int l_dtype, const void* W1,
                              const void* W2, int w_dtype, int rank, const int32_t* anchors,
                              const int32_t* draft_tokens, const float* draft_stats,
                              const float* target_stats, float temperature, int R, int gamma, int V,
                              float* conf, float* survival, void* ws, size_t ws_bytes, void* stream,
                              const uint32_t* mask) {
  if (!sizes_ok(R, gamma, V) || rank < 0 || rank > 1024) return SPEC_ERR_INVALID_ARG;
  if (!dtype_ok(l_dtype) || (rank > 0 && !dtype_ok(w_dtype))) return SPEC_ERR_UNSUPPORTED_DTYPE;
  if (!(temperature > 0.0f) || !isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
  Layout L;
  int rc = check_ws(ws, ws_bytes, SPEC_OP_TV_CONFIDENCE, R, gamma, V, rank, &L);
  if (rc != SPEC_OK) return rc;
  if (R == 0 || gamma == 0) return SPEC_OK;
  if (!U || !target || !draft_tokens || !conf) return SPEC_ERR_INVALID_ARG;
  if (rank > 0 && (!W1 || !W2 || !anchors)) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Ws w = carve(ws, L);
  const float scale = 1.0f / temperature;
  const int wdt = rank > 0 ? w_dtype : l_dtype;

  const float* tstats = target_stats;
  if (!tstats) {
    target_stats_pass(target, l_dtype, scale, R, gamma, V, nullptr, w.tstats, w, s);
    tstats = w.tstats;
  }
  RowJob j;
  memset(&j, 0, sizeof j);
  j.rows = R * gamma;
  j.map = MAP_ALL_POS;
  j.mode = MODE_STATS;
  j.R = R;
  j.gamma = gamma;
  j.V = V;
  j.scale = scale;
  j.U = U;
  j.W1 = W1;
  j.W2 = W2;
  j.rank = rank;
  j.anchors = anchors;
  j.tokens = draft_tokens;
  j.T = target;
  j.tstats = tstats;
  j.status = w.status;
  j.mask = mask;
  j.mask_words = (V + 31) / 32;
  const bool vec = vec_ok(U, target, l_dtype, V);
  const float* dstats = draft_stats;
  if (!dstats) {
    int nseg;
    if (rank == 0) {
      nseg = stream_nseg(V);
      launch_stream_partials(j, l_dtype, kStreamSeg, nseg, vec, true, false, w.pm, w.ps, w.pi,
                             grid_for((long long)j.rows * nseg, 1), s);
    } else {
      int seg;
      rc = markov_pass(j, l_dtype, wdt, w, false, s, &seg, &nseg);
      if (rc != SPEC_OK) return rc;
    }
    launch_finalize_stats(j.rows, nseg, w.pm, w.ps, w.dstats, nullptr, 1, w.status, s);
    dstats = w.dstats;
  }
  j.mode = MODE_TV;
  j.dstats = dstats;
  int nseg;
  if (rank == 0) {
    nseg = stream_nseg(V);
    launch_stream_partials(j, l_dtype, kStreamSeg, nseg, vec, true, false, w.pm, w.ps, w.pi,
                           grid_for((long long)j.rows * nseg, 1), s);
  } else {
    int seg;
    rc = markov_pass(j, l_dtype, wdt, w, false, s, &seg, &nseg);
    if (rc != SPEC_OK) return rc;
  }
  launch_tv_finalize(R, gamma, nseg, w.ps, conf, survival, s);
  return finish();
}

static int schedule_impl(const float* survival, const double* sps, int Bmax, int R, int gamma,
                         const int32_t* capacity, int32_t* lengths, int32_t* B_out,
                         double* theta_out, int32_t* B_opt_out, void* ws, size_t ws_bytes,
                         void* stream) {
  if (R < 0 || gamma < 0 || Bmax < R) return SPEC_ERR_INVALID_ARG;
  if ((long long)R * gamma > SPEC_SCHEDULE_MAX_CANDIDATES || R > SPEC_SCHEDULE_MAX_CANDIDATES)
    return SPEC_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kHeader || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0)
    return SPEC_ERR_INVALID_ARG;
  if (!sps || !B_out || !theta_out || (R > 0 && !lengths) || (R * gamma > 0 && !survival))
    return SPEC_ERR_INVALID_ARG;
  TraceScope ts(SPEC_KCLASS_OTHER, static_cast<cudaStream_t>(stream));
  const cudaError_t e = launch_schedule(survival, sps, Bmax, R, gamma, capacity, lengths, B_out,
                                        theta_out, B_opt_out, static_cast<uint32_t*>(ws),
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_schedule_prefix(const float* survival, const double* sps, int Bmax, int R, int gamma,
                         int32_t* lengths, int32_t* B_out, double* theta_out, void* ws,
                         size_t ws_bytes, void* stream) {
  return schedule_impl(survival, sps, Bmax, R, gamma, nullptr, lengths, B_out, theta_out,
                       nullptr, ws, ws_bytes, stream);
}

int spec_schedule_topk(const float* survival, const double* sps, int Bmax, int R, int gamma,
                       const int32_t* capacity, int32_t* lengths, int32_t* B_out,
                       double* theta_out, int32_t* B_opt_out, void* ws, size_t ws_bytes,
                       void* stream) {
  if (!capacity) return SPEC_ERR_INVALID_ARG;
  return schedule_impl(survival, sps, Bmax, R, gamma, capacity, lengths, B_out, theta_out,
                       B_opt_out, ws, ws_bytes, stream);
}

// The plain entry points are the no-mask case of the grammar-masked ones.

int spec_markov_propose(const void* U, int u_dtype, const void* W1, const void* W2, int w_dtype,
                        int rank, const int32_t* anchors, const float* u_draft,
                        float temperature, int R, int gamma, int V, int32_t* draft_tokens,
                        float* draft_logp, float* draft_stats, void* ws, size_t ws_bytes,
                        void* stream) {
  return markov_propose_impl(U, u_dtype, W1, W2, w_dtype, rank, anchors, u_draft, temperature, R,
                             gamma, V, draft_tokens, draft_logp, draft_stats, ws, ws_bytes,
                             stream, nullptr);
}

int spec_mtp_greedy(const void* D, const void* target, int dtype, const int32_t* lengths, int R,
                    int gamma, int V, int32_t* draft_tokens, int32_t* accept_len,
                    int32_t* out_tokens, int32_t* next_anchor, void* ws, size_t ws_bytes,
                    void* stream) {
  if (!sizes_ok(R, gamma, V)) return SPEC_ERR_INVALID_ARG;
  if (!dtype_ok(dtype)) return SPEC_ERR_UNSUPPORTED_DTYPE;
  Layout L;
  int rc = check_ws(ws, ws_bytes, SPEC_OP_MTP_GREEDY, R, gamma, V, 0, &L);
  if (rc != SPEC_OK) return rc;
  if (R == 0) return SPEC_OK;
  if (!target || !accept_len || (gamma > 0 && (!D || !draft_tokens))) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mtp_greedy_supported(dtype, R, gamma, V, D, target)) {
    const Ws w = carve(ws, L);
    if (launch_mtp_greedy(dtype, D, target, R, gamma, V, lengths, draft_tokens, accept_len,
                          out_tokens, next_anchor, w.pm, w.pi, w.status, s) != cudaSuccess)
      return SPEC_ERR_CUDA;
    return finish();
  }
  if (gamma > 0) {
    rc = markov_propose_impl(D, dtype, nullptr, nullptr, dtype, 0, nullptr, nullptr, 0.0f, R,
                             gamma, V, draft_tokens, nullptr, nullptr, ws, ws_bytes, stream,
                             nullptr);
    if (rc != SPEC_OK) return rc;
  }
  return verify_greedy_impl(target, dtype, draft_tokens, lengths, nullptr, R, gamma, V,
                            accept_len, out_tokens, next_anchor, ws, ws_bytes, stream);
}

int spec_markov_propose_masked(const void* U, int u_dtype, const void* W1, const void* W2,
                               int w_dtype, int rank, const int32_t* anchors,
                               const float* u_draft, float temperature, int R, int gamma, int V,
                               int32_t* draft_tokens, float* draft_logp, float* draft_stats,
                               const uint32_t* allowed, void* ws, size_t ws_bytes,
                               void* stream) {
  return markov_propose_impl(U, u_dtype, W1, W2, w_dtype, rank, anchors, u_draft, temperature, R,
                             gamma, V, draft_tokens, draft_logp, draft_stats, ws, ws_bytes,
                             stream, allowed);
}

int spec_markov_propose_target_stats(const void* U, int l_dtype, const void* W1, const void* W2,
                                     int w_dtype, int rank, const int32_t* anchors,
                                     const float* u_draft, float temperature, int R, int gamma,
                                     int V, int32_t* draft_tokens, float* draft_logp,
                                     float* draft_stats, const void* target, float* target_stats,
                                     void* ws, size_t ws_bytes, void* stream) {
  if (!target) return SPEC_ERR_INVALID_ARG;
  return markov_propose_impl(U, l_dtype, W1, W2, w_dtype, rank, anchors, u_draft, temperature, R,
                             gamma, V, draft_tokens, draft_logp, draft_stats, ws, ws_bytes,
                             stream, nullptr, target, target_stats);
}

int spec_verify_rejection(const void* target, const void* U, int l_dtype, const void* W1,
                          const void* W2, int w_dtype, int rank, const int32_t* anchors,
                          const int32_t* draft_tokens, const float* draft_logp,
                          const float* draft_stats, const float* target_stats,
                          const float* u_accept, const float* u_resid, float temperature,
                          const int32_t* lengths, int R, int gamma, int V, int32_t* accept_len,
                          int32_t* out_tokens, int32_t* next_anchor, void* ws, size_t ws_bytes,
                          void* stream) {
  return verify_rejection_impl(target, U, l_dtype, W1, W2, w_dtype, rank, anchors, draft_tokens,
                               draft_logp, draft_stats, target_stats, u_accept, u_resid,
                               temperature, lengths, R, gamma, V, accept_len, out_tokens,
                               next_anchor, ws, ws_bytes, stream, nullptr);
}

int spec_verify_rejection_masked(const void* target, const void* U, int l_dtype, const void* W1,
                                 const void* W2, int w_dtype, int rank, const int32_t* anchors,
                                 const int32_t* draft_tokens, const float* draft_logp,
                                 const float* draft_stats, const float* target_stats,
                                 const float* u_accept, const float* u_resid, float temperature,
                                 const int32_t* lengths, int R, int gamma, int V,
                                 int32_t* accept_len, int32_t* out_tokens, int32_t* next_anchor,
                                 const uint32_t* allowed, void* ws, size_t ws_bytes,
                                 void* stream) {
  return verify_rejection_impl(target, U, l_dtype, W1, W2, w_dtype, rank, anchors, draft_tokens,
                               draft_logp, draft_stats, target_stats, u_accept, u_resid,
                               temperature, lengths, R, gamma, V, accept_len, out_tokens,
                               next_anchor, ws, ws_bytes, stream, allowed);
}

int spec_verify_rejection_flat(const void* target, const void* U, int l_dtype, const void* W1,
                               const void* W2, int w_dtype, int rank, const int32_t* anchors,
                               const int32_t* draft_tokens, const float* draft_logp,
                               const float* draft_stats, const float* target_stats,
                               const float* u_accept, const float* u_resid, float temperature,
                               const int32_t* lengths, const int32_t* offsets, int R, int gamma,
                               int V, int32_t* accept_len, int32_t* out_tokens,
                               int32_t* next_anchor, const uint32_t* allowed, void* ws,
                               size_t ws_bytes, void* stream) {
  if (R > 0 && (!lengths || !offsets)) return SPEC_ERR_INVALID_ARG;
  return verify_rejection_impl(target, U, l_dtype, W1, W2, w_dtype, rank, anchors, draft_tokens,
                               draft_logp, draft_stats, target_stats, u_accept, u_resid,
                               temperature, lengths, R, gamma, V, accept_len, out_tokens,
                               next_anchor, ws, ws_bytes, stream, allowed, offsets);
}

int spec_tv_confidence(const void* U, const void* target, int l_dtype, const void* W1,
                       const void* W2, int w_dtype, int rank, const int32_t* anchors,
                       const int32_t* draft_tokens, const float* draft_stats,
                       const float* target_stats, float temperature, int R, int gamma, int V,
                       float* conf, float* survival, void* ws, size_t ws_bytes, void* stream) {
  return tv_confidence_impl(U, target, l_dtype, W1, W2, w_dtype, rank, anchors, draft_tokens,
                            draft_stats, target_stats, temperature, R, gamma, V, conf, survival,
                            ws, ws_bytes, stream, nullptr);
}

int spec_tv_confidence_masked(const void* U, const void* target, int l_dtype, const void* W1,
                              const void* W2, int w_dtype, int rank, const int32_t* anchors,
                              const int32_t* draft_tokens, const float* draft_stats,
                              const float* target_stats, float temperature, int R, int gamma,
                              int V, float* conf, float* survival, const uint32_t* allowed,
                              void* ws, size_t ws_bytes, void* stream) {
  return tv_confidence_impl(U, target, l_dtype, W1, W2, w_dtype, rank, anchors, draft_tokens,
                            draft_stats, target_stats, temperature, R, gamma, V, conf, survival,
                            ws, ws_bytes, stream, allowed);
}

}  // extern "C"
