// kernels.h -- host-side launchers of the libspecmarkov kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace spec {

// Number of vocabulary columns per partial of the Markov producers (one epilogue half-tile).
constexpr int kMarkovSeg = 64;
// Number of vocabulary columns per partial of the rank-0 streaming producer.
constexpr int kStreamSeg = 32768;

// Per-row outputs of a select pass.
struct SelectOut {
  int kind;              // 0: draft proposal at position k, 1: final token of rejection verify
  int32_t* tokens;       // kind 0: draft_tokens [R, gamma]; kind 1: out_tokens [R, gamma+1]
  float* logp;           // kind 0, optional
  float* stats;          // kind 0, optional
  int32_t* next_anchor;  // kind 1, optional
  const float* uni;      // uniforms, indexed row * uni_stride + uni_offset
  int uni_stride, uni_offset;
  int greedy;
  // optional: the Markov embedding; the row of each drawn token (w1_row_bytes, a multiple of
  // 16) is pulled into L2 for the next position's A-operand gather
  const void* w1;
  int w1_row_bytes;
};

// Optional L2 prefetch of the W1 rows that the residual pass will gather (the previous token
// of each request's final row); w1 == nullptr disables it.
struct RowPrefetch {
  const void* w1;
  int row_bytes;
  const int32_t* anchors;
};

void launch_stream_partials(const RowJob& j, int dtype, int seg, int nseg, bool vec, bool sum,
                            bool argmax, float* pm, float* ps, int* pi, int grid,
                            cudaStream_t s);
void launch_ffma_partials(const RowJob& j, int udt, int wdt, int nseg, bool argmax, float* pm,
                          float* ps, int* pi, int grid, cudaStream_t s);
void launch_select(const RowJob& j, int udt, int wdt, int seg, int nseg, const float* pm,
                   const float* ps, const int* pi, const SelectOut& o, cudaStream_t s);
void launch_finalize_stats(int rows, int nseg, const float* pm, const float* ps, float* stats,
                           const int32_t* lengths, int rows_per_req, uint32_t* status,
                           cudaStream_t s);
void launch_greedy_scan(int R, int gamma, const int* amax, const int32_t* tokens,
                        const int32_t* lengths, const int32_t* toff, int32_t* accept_len,
                        int32_t* out_tokens, int32_t* next_anchor, uint32_t* status,
                        cudaStream_t s);
// Per-row (m, log Z) and/or first argmax of target rows (MAP_TARGET job), one block per row.
void launch_row_stats(const RowJob& j, int dtype, bool vec, float* stats, int* argmax,
                      cudaStream_t s);
void launch_accept(int dtype, int R, int gamma, int V, float scale, const void* T,
                   const float* tstats, const int32_t* tokens, const float* dlogp,
                   const float* u_accept, const int32_t* lengths, const int32_t* toff,
                   int32_t* final_n, int32_t* final_kind, int32_t* accept_len,
                   int32_t* out_tokens, uint32_t* status, RowPrefetch pf, bool chained,
                   cudaStream_t s);
void launch_tv_finalize(int R, int gamma, int nseg, const float* ps, float* conf, float* survival,
                        cudaStream_t s);
cudaError_t launch_schedule(const float* survival, const double* sps, int Bmax, int R, int gamma,
                            const int32_t* b_cap, int32_t* lengths, int32_t* B_out,
                            double* theta_out, int32_t* B_opt_out, uint32_t* status,
                            cudaStream_t s);
size_t schedule_smem_bytes(int R, int gamma);
// Flattened verify batch layout from per-request lengths (offsets [R+1], optional row markers).
void launch_flat_layout(const int32_t* lengths, int R, int gamma, int32_t* offsets,
                        int32_t* row_req, int32_t* row_pos, uint32_t* status, cudaStream_t s);
// Rows (r, i <= l_r) of a padded [R, gamma+1] array of row_bytes-byte rows to packed rows
// offsets[r] + i (row_bytes a multiple of 4).
void launch_flat_pack(const void* src, int row_bytes, const int32_t* lengths,
                      const int32_t* offsets, int R, int gamma, void* dst, uint32_t* status,
                      cudaStream_t s);

// tcgen05 Markov producer (markov_tc.cu). Returns false when the shape is not supported
// (the caller then uses the CUDA-core producer).
bool markov_tc_supported(int udt, int wdt, int rank, int V, const void* U, const void* T,
                         const void* W1, const void* W2);
cudaError_t launch_markov_tc(const RowJob& j, float* pm, float* ps, int* pi, bool argmax,
                             cudaStream_t s);
// The whole Markov proposal (all positions, selects included) in one persistent tcgen05 launch
// (markov_propose.cu); `sync` is the workspace's counter area, zero on entry and on return.
bool markov_propose_tc_supported(int udt, int wdt, int rank, int R, int gamma, int V,
                                 const void* U, const void* W1, const void* W2);
// With `target` (bf16 [R * (gamma + 1), V]) the same launch also writes the target rows'
// softmax normalisers (m, log Z) of target * tscale into tstats.
cudaError_t launch_markov_propose_tc(const RowJob& j, const SelectOut& o, float* pm, float* ps,
                                     int* pi, bool argmax, uint32_t* sync, cudaStream_t s,
                                     const void* target = nullptr, float* tstats = nullptr,
                                     float tscale = 1.0f);
// Workspace bytes [kSyncOffset, kSyncOffset + kSyncBytes): inter-CTA counters of the persistent
// proposal, at a fixed place whatever the problem size, zeroed by spec_workspace_init.
constexpr size_t kSyncOffset = 256;
constexpr size_t kSyncBytes = 8192;
// CTAs of the persistent proposal at most (the coarse partials of its select, two per CTA and
// row, are sized for this many).
constexpr int kMaxPropGrid = 256;
// A 2-D or 3-D bf16 tensor map with a 128-byte swizzle (false if it cannot be encoded).
bool make_tensor_map_bf16(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                          const cuuint64_t* strides_bytes, const cuuint32_t* box);
// Consume the test request that makes the next tensor-core launch never load its first W2
// tile (spec_test_stall_next_markov).
int take_stall_request();
// Vocabulary columns per partial written by the tcgen05 producer in pass mode `mode`.
int markov_tc_seg(int mode);
// MTP/NextN greedy proposal + greedy verification (mtp.cu): one streaming launch takes the
// argmax of every draft and target row in kMtpChunk-element items (pm / pi: one partial per
// item, R * (2 gamma + 1) * cdiv(V, kMtpChunk) of them), a chained launch merges them per
// request and runs the scan.
constexpr int kMtpChunk = 4096;
constexpr int kMtpMaxGamma = 1024;
bool mtp_greedy_supported(int dtype, int R, int gamma, int V, const void* D, const void* T);
cudaError_t launch_mtp_greedy(int dtype, const void* D, const void* T, int R, int gamma, int V,
                              const int32_t* lengths, int32_t* draft_tokens, int32_t* accept_len,
                              int32_t* out_tokens, int32_t* next_anchor, float* pm, int* pi,
                              uint32_t* status, cudaStream_t s);
// Smallest partial segment any Markov producer writes (sizes the workspace).
constexpr int kMarkovMinSeg = 32;

int num_sms();

// Tracing hooks around every launch (api.cu): count the launch and record the attached begin /
// end events of its kernel class on the launch stream.
void trace_begin(int kclass, cudaStream_t s);
void trace_end(int kclass, cudaStream_t s);

// Whether any kernel class has caller-owned trace events attached. Chained launches are then
// issued plainly, so that every recorded interval spans exactly one kernel.
bool trace_active();

// Launch of kernel k on stream s. With `chained` it is a programmatic dependent launch: k is
// scheduled as the blocks of the previous kernel on the stream exit, without waiting for that
// kernel's completion, and must call grid_dep_wait before it touches what that kernel or an
// earlier one of the same call writes or reads. Only the kernels of a call after its first
// launch are chained, so what a chained kernel reads before its wait (inputs of the call that
// no kernel of the call writes) was finished before the call's first kernel began.
template <typename... P, typename... A>
cudaError_t launch_kernel(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          bool chained, A&&... args) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = &attr;
  cfg.numAttrs = chained && !trace_active() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, static_cast<A&&>(args)...);
}

struct TraceScope {
  int kclass;
  cudaStream_t s;
  TraceScope(int k, cudaStream_t st) : kclass(k), s(st) { trace_begin(k, st); }
  ~TraceScope() { trace_end(kclass, s); }
};

}  // namespace spec
