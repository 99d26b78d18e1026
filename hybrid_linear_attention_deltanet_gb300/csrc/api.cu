// C ABI of the library: host-side argument checks, scratch management and
// dispatch to the kernels.  Declarations and contracts: include/gdn.h.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "backward.cuh"
#include "gdn_internal.cuh"
#include "../../include/gdn_testing.h"

namespace gdn {

// Device status word (first device-side error code since the last read).
__device__ unsigned g_status_word = 0;

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {

constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;

// Per-device stream-ordered pool for the prefill scratch.  Its release
// threshold keeps freed scratch mapped for later calls: the default pool
// hands memory back to the system at every synchronisation, and mapping a
// few hundred MB again costs about as much as the prefill itself.  The pool
// holds the largest scratch any call needed until the process exits.
cudaMemPool_t g_scratch_pool[kMaxDevices] = {};
std::mutex g_pool_mu;

cudaMemPool_t scratch_pool() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  if (!g_scratch_pool[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
    uint64_t keep = ~0ull;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return nullptr;
    }
    g_scratch_pool[dev] = pool;
  }
  return g_scratch_pool[dev];
}

// This device's pool if a call has created it (nullptr otherwise).
cudaMemPool_t existing_scratch_pool(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  return g_scratch_pool[dev];
}

}  // namespace

cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t stream) {
  cudaMemPool_t pool = scratch_pool();
  if (!pool) return cudaErrorMemoryAllocation;
  return cudaMallocFromPoolAsync(p, bytes, pool, stream);
}

cudaError_t scratch_free(void* p, cudaStream_t stream) {
  return p ? cudaFreeAsync(p, stream) : cudaSuccess;
}

// Address of this device's status word, looked up once per device with that
// device current.
unsigned* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = (unsigned*)p;
  }
  return g_status_ptr[dev];
}

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};
Range span(const void* p, size_t bytes) { return {(uintptr_t)p, (uintptr_t)p + bytes}; }
bool overlaps(Range a, Range b) {
  return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

// cu_seqlens -> exclusive prefix of per-sequence chunk counts, with the
// monotonicity / end checks.  One CTA; N may be large, so it loops in tiles.
__global__ void __launch_bounds__(1024)
chunk_offsets_kernel(const int32_t* __restrict__ cu, int32_t N, int64_t T_total,
                     int32_t* __restrict__ chunk_off, unsigned* status) {
  __shared__ int bad;
  __shared__ int64_t carry;
  __shared__ int64_t warp_tot[32];
  if (threadIdx.x == 0) {
    bad = (cu[0] != 0 || (int64_t)cu[N] != T_total) ? 1 : 0;
    carry = 0;
  }
  __syncthreads();
  for (int n = threadIdx.x; n < N; n += blockDim.x)
    if (cu[n + 1] < cu[n]) bad = 1;
  __syncthreads();
  if (bad) {
    for (int n = threadIdx.x; n <= N; n += blockDim.x) chunk_off[n] = 0;
    if (threadIdx.x == 0) flag_status(status, GDN_ERR_BAD_SEQLENS);
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = 0; base < N; base += blockDim.x) {
    const int n = base + threadIdx.x;
    int64_t c = n < N ? ((int64_t)cu[n + 1] - cu[n] + kC - 1) / kC : 0;
    int64_t x = c;  // inclusive warp scan
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int64_t w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int64_t before = carry + (warp ? warp_tot[warp - 1] : 0) + x - c;
    if (n < N) chunk_off[n] = (int32_t)before;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = before + c;
    __syncthreads();
  }
  if (threadIdx.x == 0) chunk_off[N] = (int32_t)carry;
}

}  // namespace

cudaError_t launch_chunk_offsets(const int32_t* cu_seqlens, int32_t N, int64_t T_total,
                                 int32_t* chunk_off, unsigned* status, cudaStream_t stream) {
  chunk_offsets_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, N, T_total, chunk_off, status);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace gdn

using namespace gdn;

extern "C" {

}  // extern "C"

namespace gdn {

// Scratch of one prefill call.  Plain form: the packed batch's chunk
// offsets, then the path's per-chunk scratch (bf16 I/O: the tensor-core
// path; fp32: the CUDA-core path); zero when the call needs none.  Segmented
// form (a sequence may be long, or the caller fixed the segment count): the
// plan's layout.
bool takes_long_form(int64_t seqlen, int32_t forced_P) {
  return forced_P > 0 || long_form_applies(seqlen);
}

size_t prefill_scratch_bytes(int32_t batch, int64_t seqlen, int32_t heads, int32_t dv,
                             int32_t io_dtype, bool varlen, int32_t forced_P) {
  if (takes_long_form(seqlen, forced_P))
    return plan_long(batch, seqlen, varlen, heads, dv, io_dtype, forced_P).bytes;
  const int64_t T_total = varlen ? seqlen : (int64_t)batch * seqlen;
  const int64_t max_chunks = max_chunks_bound(batch, T_total, varlen, seqlen);
  const size_t off_bytes = varlen ? align_up(((size_t)batch + 1) * 4, 256) : 0;
  const size_t work_bytes = io_dtype == GDN_BF16
                                ? prefill_tc_scratch_bytes(max_chunks, heads, dv)
                                : prefill_simt_scratch_bytes(max_chunks, heads, dv);
  return off_bytes + work_bytes;
}

// The prefill of a validated problem (a: the caller's map, tensors and
// status word) with `scratch` of prefill_scratch_bytes(...) bytes: the
// segmented form, or the chunk offsets of a packed batch and the path's
// kernels.
cudaError_t launch_prefill_any(PrefillLaunch a, int32_t io_dtype, int64_t seqlen,
                               int32_t forced_P, void* scratch, cudaStream_t stream) {
  const bool varlen = a.map.cu_seqlens != nullptr;
  if (takes_long_form(seqlen, forced_P)) {
    a.scratch = scratch;
    return launch_prefill_long(a, io_dtype,
                               plan_long(a.map.N, seqlen, varlen, a.H, a.dv, io_dtype, forced_P),
                               forced_P, stream);
  }
  const size_t off_bytes = varlen ? align_up(((size_t)a.map.N + 1) * 4, 256) : 0;
  a.scratch = (char*)scratch + off_bytes;
  if (varlen) {
    a.map.chunk_off = (int32_t*)scratch;
    const int64_t T_total = a.map.T;
    const cudaError_t e =
        launch_chunk_offsets(a.map.cu_seqlens, a.map.N, T_total, (int32_t*)scratch, a.status, stream);
    if (e != cudaSuccess) return e;
  }
  return io_dtype == GDN_BF16 ? launch_prefill_tc(a, stream)
                              : launch_prefill_simt(a, io_dtype, stream);
}

namespace {

bool prefill_shape_ok(int32_t batch, int64_t seqlen, int32_t heads, int32_t dk, int32_t dv,
                      int32_t io_dtype) {
  return batch >= 1 && seqlen >= 0 && heads >= 1 && dk == kDK && supported_dv(dv) &&
         (io_dtype == GDN_F32 || io_dtype == GDN_BF16);
}

// A caller's workspace: large enough, 256-byte aligned, overlapping nothing
// the call reads or writes.
int check_workspace(const void* ws, size_t ws_bytes, size_t need, const Range* used, int n_used) {
  if (need == 0) return GDN_OK;
  if (!ws || ws_bytes < need) return GDN_ERR_INVALID_ARG;
  if ((uintptr_t)ws & 255u) return GDN_ERR_ALIGNMENT;
  const Range w = span(ws, need);
  for (int i = 0; i < n_used; ++i)
    if (overlaps(w, used[i])) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

// gdn_prefill, gdn_prefill_scan and their _ws forms: scratch from the
// caller's workspace when use_ws, else stream-ordered from the library's
// pool; forced_P > 0 fixes the segment count of every sequence.
int prefill_common(const void* q, const void* k, const void* v, const float* alpha,
                   const float* beta, const float* S0, const int32_t* cu_seqlens, void* out,
                   float* S_final, int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                   int32_t dv, int32_t io_dtype, int32_t forced_P, cudaStream_t stream,
                   bool use_ws, void* ws, size_t ws_bytes) {
  if (batch < 1 || seqlen < 0 || heads < 1 || forced_P < 0) return GDN_ERR_INVALID_ARG;
  const bool varlen = cu_seqlens != nullptr;
  const int64_t T_total = varlen ? seqlen : (int64_t)batch * seqlen;
  // token tensors may be empty (and then null) only when there are no tokens
  if (T_total > 0 && (!q || !k || !v || !alpha || !beta || !out)) return GDN_ERR_INVALID_ARG;
  if (io_dtype != GDN_F32 && io_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if (dk != kDK || !supported_dv(dv)) return GDN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned4(alpha) || !aligned4(beta) ||
      !aligned16(out) || !aligned16(S0) || !aligned16(S_final) || !aligned4(cu_seqlens))
    return GDN_ERR_ALIGNMENT;
  const bool long_form = takes_long_form(seqlen, forced_P);
  // 32-bit offsets (packed batches, the segmented form) and token coordinates
  // (tensor-core path)
  if ((varlen || long_form || io_dtype == GDN_BF16) && T_total > 0x7fffffffLL)
    return GDN_ERR_UNSUPPORTED;
  LongPlan plan;
  if (long_form) {
    plan = plan_long(batch, seqlen, varlen, heads, dv, io_dtype, forced_P);
    if (plan.n_slots * 2 > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  }
  const size_t es = io_dtype == GDN_BF16 ? 2 : 4;
  const size_t n_tok_h = (size_t)T_total * heads;
  const size_t state_bytes = (size_t)batch * heads * dv * dk * sizeof(float);
  const Range used[] = {span(q, n_tok_h * dk * es), span(k, n_tok_h * dk * es),
                        span(v, n_tok_h * dv * es), span(alpha, n_tok_h * 4),
                        span(beta, n_tok_h * 4),
                        span(S0, S0 ? state_bytes : 0),
                        span(cu_seqlens, varlen ? ((size_t)batch + 1) * 4 : 0),
                        span(out, n_tok_h * dv * es),
                        span(S_final, S_final ? state_bytes : 0)};
  const int n_in = 7;
  const Range& r_out = used[7];
  const Range& r_sf = used[8];
  for (int i = 0; i < n_in; ++i)
    if (overlaps(used[i], r_out) || overlaps(used[i], r_sf)) return GDN_ERR_INVALID_ARG;
  if (overlaps(r_out, r_sf)) return GDN_ERR_INVALID_ARG;
  const size_t need = long_form ? plan.bytes
                                : prefill_scratch_bytes(batch, seqlen, heads, dv, io_dtype,
                                                        varlen, 0);
  if (use_ws) {
    const int rc = check_workspace(ws, ws_bytes, need, used, 9);
    if (rc != GDN_OK) return rc;
  }

  unsigned* status = status_ptr();
  if (!status) return GDN_ERR_CUDA;

  PrefillLaunch a{};
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.S0 = S0;
  a.out = out; a.S_final = S_final; a.H = heads; a.status = status;
  a.map.cu_seqlens = cu_seqlens;
  a.map.N = batch;
  a.map.T = varlen ? T_total : seqlen;
  a.map.chunks_per_seq = varlen ? 0 : (seqlen + kC - 1) / kC;
  a.max_chunks = max_chunks_bound(batch, T_total, varlen, seqlen);

  // bf16 I/O runs on the tensor cores, fp32 I/O on the CUDA cores
  const bool tc = io_dtype == GDN_BF16;
  a.dv = dv;
  a.allow_overlap = true;
  void* scratch = use_ws ? ws : nullptr;
  if (!use_ws && need > 0 &&
      (!scratch_pool() ||
       cudaMallocFromPoolAsync(&scratch, need, scratch_pool(), stream) != cudaSuccess))
    return GDN_ERR_CUDA;
  (void)tc;
  const cudaError_t e = launch_prefill_any(a, io_dtype, seqlen, forced_P, scratch, stream);
  const cudaError_t ef = (!use_ws && scratch) ? cudaFreeAsync(scratch, stream) : cudaSuccess;
  return (e == cudaSuccess && ef == cudaSuccess) ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace
}  // namespace gdn

extern "C" {

int gdn_prefill(const void* q, const void* k, const void* v, const float* alpha,
                const float* beta, const float* S0, const int32_t* cu_seqlens, void* out,
                float* S_final, int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                int32_t dv, int32_t io_dtype, gdn_stream_t stream) {
  return prefill_common(q, k, v, alpha, beta, S0, cu_seqlens, out, S_final, batch, seqlen, heads,
                        dk, dv, io_dtype, 0, (cudaStream_t)stream, false, nullptr, 0);
}

size_t gdn_prefill_workspace_size(int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                                  int32_t dv, int32_t io_dtype, int32_t varlen) {
  if (!prefill_shape_ok(batch, seqlen, heads, dk, dv, io_dtype)) return SIZE_MAX;
  return prefill_scratch_bytes(batch, seqlen, heads, dv, io_dtype, varlen != 0, 0);
}

int gdn_prefill_ws(const void* q, const void* k, const void* v, const float* alpha,
                   const float* beta, const float* S0, const int32_t* cu_seqlens, void* out,
                   float* S_final, int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                   int32_t dv, int32_t io_dtype, void* workspace, size_t workspace_bytes,
                   gdn_stream_t stream) {
  return prefill_common(q, k, v, alpha, beta, S0, cu_seqlens, out, S_final, batch, seqlen, heads,
                        dk, dv, io_dtype, 0, (cudaStream_t)stream, true, workspace,
                        workspace_bytes);
}

int gdn_prefill_scan(const void* q, const void* k, const void* v, const float* alpha,
                     const float* beta, const float* S0, const int32_t* cu_seqlens, void* out,
                     float* S_final, int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                     int32_t dv, int32_t io_dtype, int32_t segments, gdn_stream_t stream) {
  if (segments < 1) return GDN_ERR_INVALID_ARG;
  return prefill_common(q, k, v, alpha, beta, S0, cu_seqlens, out, S_final, batch, seqlen, heads,
                        dk, dv, io_dtype, segments, (cudaStream_t)stream, false, nullptr, 0);
}

size_t gdn_prefill_scan_workspace_size(int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                                       int32_t dv, int32_t io_dtype, int32_t varlen,
                                       int32_t segments) {
  if (!prefill_shape_ok(batch, seqlen, heads, dk, dv, io_dtype) || segments < 1) return SIZE_MAX;
  return prefill_scratch_bytes(batch, seqlen, heads, dv, io_dtype, varlen != 0, segments);
}

int gdn_prefill_scan_ws(const void* q, const void* k, const void* v, const float* alpha,
                        const float* beta, const float* S0, const int32_t* cu_seqlens, void* out,
                        float* S_final, int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                        int32_t dv, int32_t io_dtype, int32_t segments, void* workspace,
                        size_t workspace_bytes, gdn_stream_t stream) {
  if (segments < 1) return GDN_ERR_INVALID_ARG;
  return prefill_common(q, k, v, alpha, beta, S0, cu_seqlens, out, S_final, batch, seqlen, heads,
                        dk, dv, io_dtype, segments, (cudaStream_t)stream, true, workspace,
                        workspace_bytes);
}

}  // extern "C"

namespace gdn {
namespace {

size_t backward_scratch_bytes(int32_t batch, int64_t seqlen, int32_t heads, int32_t dv,
                              int32_t io_dtype, bool varlen) {
  const int64_t T_total = varlen ? seqlen : (int64_t)batch * seqlen;
  const int64_t max_chunks = max_chunks_bound(batch, T_total, varlen, seqlen);
  const size_t off_bytes = varlen ? align_up(((size_t)batch + 1) * 4, 1024) : 0;
  return off_bytes + prefill_backward_scratch_bytes(max_chunks, heads, dv, T_total, io_dtype);
}

// gdn_prefill_backward and gdn_prefill_backward_ws (workspace 1024-byte aligned)
int backward_common(const void* q, const void* k, const void* v, const float* alpha,
                    const float* beta, const float* S0, const int32_t* cu_seqlens,
                    const void* dout, const float* dS_final, void* dq, void* dk, void* dv_,
                    float* dalpha, float* dbeta, float* dS0, int32_t batch, int64_t seqlen,
                    int32_t heads, int32_t dk_, int32_t dv, int32_t io_dtype, cudaStream_t stream,
                    bool use_ws, void* ws, size_t ws_bytes) {
  if (batch < 1 || seqlen < 0 || heads < 1) return GDN_ERR_INVALID_ARG;
  const bool varlen = cu_seqlens != nullptr;
  const int64_t T_total = varlen ? seqlen : (int64_t)batch * seqlen;
  if (T_total > 0 && (!q || !k || !v || !alpha || !beta || !dout || !dq || !dk || !dv_ ||
                      !dalpha || !dbeta))
    return GDN_ERR_INVALID_ARG;
  if (io_dtype != GDN_F32 && io_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if (dk_ != kDK || !supported_dv(dv)) return GDN_ERR_UNSUPPORTED;
  const void* a16[] = {q, k, v, dout, dq, dk, dv_, S0, dS_final, dS0};
  for (const void* p : a16)
    if (!aligned16(p)) return GDN_ERR_ALIGNMENT;
  if (!aligned4(alpha) || !aligned4(beta) || !aligned4(dalpha) || !aligned4(dbeta) ||
      !aligned4(cu_seqlens))
    return GDN_ERR_ALIGNMENT;
  if ((varlen || io_dtype == GDN_BF16) && T_total > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  const size_t es = io_dtype == GDN_BF16 ? 2 : 4;
  const size_t nth = (size_t)T_total * heads;
  const size_t state_bytes = (size_t)batch * heads * dv * dk_ * sizeof(float);
  const Range all[] = {span(q, nth * dk_ * es), span(k, nth * dk_ * es), span(v, nth * dv * es),
                       span(alpha, nth * 4), span(beta, nth * 4), span(S0, S0 ? state_bytes : 0),
                       span(cu_seqlens, varlen ? ((size_t)batch + 1) * 4 : 0),
                       span(dout, nth * dv * es), span(dS_final, dS_final ? state_bytes : 0),
                       span(dq, nth * dk_ * es), span(dk, nth * dk_ * es),
                       span(dv_, nth * dv * es), span(dalpha, nth * 4), span(dbeta, nth * 4),
                       span(dS0, dS0 ? state_bytes : 0)};
  const int n_in = 9, n_all = 15;
  for (int o = n_in; o < n_all; ++o) {
    for (int r = 0; r < n_in; ++r)
      if (overlaps(all[r], all[o])) return GDN_ERR_INVALID_ARG;
    for (int o2 = n_in; o2 < n_all; ++o2)
      if (o2 != o && overlaps(all[o], all[o2])) return GDN_ERR_INVALID_ARG;
  }
  const int64_t max_chunks = max_chunks_bound(batch, T_total, varlen, seqlen);
  if (max_chunks * heads > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;   // grid bound
  const size_t need = backward_scratch_bytes(batch, seqlen, heads, dv, io_dtype, varlen);
  if (use_ws) {
    if (ws && ((uintptr_t)ws & 1023u)) return GDN_ERR_ALIGNMENT;
    const int rc = check_workspace(ws, ws_bytes, need, all, n_all);
    if (rc != GDN_OK) return rc;
  }
  unsigned* status = status_ptr();
  if (!status) return GDN_ERR_CUDA;
  PrefillLaunch a{};
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.S0 = S0; a.H = heads;
  a.status = status; a.dv = dv;
  // the backward's scratch starts 1024-byte aligned (the tensor-core forward
  // it may run stages images with bulk copies)
  a.map.cu_seqlens = cu_seqlens;
  a.map.N = batch;
  a.map.T = varlen ? T_total : seqlen;
  a.map.chunks_per_seq = varlen ? 0 : (seqlen + kC - 1) / kC;
  a.max_chunks = max_chunks;
  const size_t off_bytes = varlen ? align_up(((size_t)batch + 1) * 4, 1024) : 0;
  void* scratch = use_ws ? ws : nullptr;
  if (!use_ws && (!scratch_pool() ||
                  cudaMallocFromPoolAsync(&scratch, need, scratch_pool(), stream) != cudaSuccess))
    return GDN_ERR_CUDA;
  a.scratch = (char*)scratch + off_bytes;
  cudaError_t e = cudaSuccess;
  if (varlen) {
    a.map.chunk_off = (int32_t*)scratch;
    e = launch_chunk_offsets(cu_seqlens, batch, T_total, (int32_t*)scratch, status, stream);
  }
  if (e == cudaSuccess)
    e = launch_prefill_backward(a, dout, dS_final, dq, dk, dv_, dalpha, dbeta, dS0, io_dtype,
                                stream);
  const cudaError_t ef = use_ws ? cudaSuccess : cudaFreeAsync(scratch, stream);
  return (e == cudaSuccess && ef == cudaSuccess) ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace
}  // namespace gdn

extern "C" {

int gdn_prefill_backward(const void* q, const void* k, const void* v, const float* alpha,
                         const float* beta, const float* S0, const int32_t* cu_seqlens,
                         const void* dout, const float* dS_final, void* dq, void* dk, void* dv_,
                         float* dalpha, float* dbeta, float* dS0, int32_t batch, int64_t seqlen,
                         int32_t heads, int32_t dk_, int32_t dv, int32_t io_dtype,
                         gdn_stream_t stream) {
  return backward_common(q, k, v, alpha, beta, S0, cu_seqlens, dout, dS_final, dq, dk, dv_,
                         dalpha, dbeta, dS0, batch, seqlen, heads, dk_, dv, io_dtype,
                         (cudaStream_t)stream, false, nullptr, 0);
}

size_t gdn_prefill_backward_workspace_size(int32_t batch, int64_t seqlen, int32_t heads,
                                           int32_t dk, int32_t dv, int32_t io_dtype,
                                           int32_t varlen) {
  if (batch < 1 || seqlen < 0 || heads < 1 || dk != kDK || !supported_dv(dv) ||
      (io_dtype != GDN_F32 && io_dtype != GDN_BF16))
    return SIZE_MAX;
  return backward_scratch_bytes(batch, seqlen, heads, dv, io_dtype, varlen != 0);
}

int gdn_prefill_backward_ws(const void* q, const void* k, const void* v, const float* alpha,
                            const float* beta, const float* S0, const int32_t* cu_seqlens,
                            const void* dout, const float* dS_final, void* dq, void* dk,
                            void* dv_, float* dalpha, float* dbeta, float* dS0, int32_t batch,
                            int64_t seqlen, int32_t heads, int32_t dk_, int32_t dv,
                            int32_t io_dtype, void* workspace, size_t workspace_bytes,
                            gdn_stream_t stream) {
  return backward_common(q, k, v, alpha, beta, S0, cu_seqlens, dout, dS_final, dq, dk, dv_,
                         dalpha, dbeta, dS0, batch, seqlen, heads, dk_, dv, io_dtype,
                         (cudaStream_t)stream, true, workspace, workspace_bytes);
}

int gdn_release_scratch(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  cudaMemPool_t pool = existing_scratch_pool(dev);
  if (!pool) return GDN_OK;
  // the pool only returns memory whose frees have completed: finish every
  // stream's work on this device first
  if (cudaDeviceSynchronize() != cudaSuccess) return GDN_ERR_CUDA;
  return cudaMemPoolTrimTo(pool, 0) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_testing_scratch_reserved(uint64_t* bytes) {
  if (!bytes) return GDN_ERR_INVALID_ARG;
  *bytes = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  cudaMemPool_t pool = existing_scratch_pool(dev);
  if (!pool) return GDN_OK;
  uint64_t v = 0;
  if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &v) != cudaSuccess)
    return GDN_ERR_CUDA;
  *bytes = v;
  return GDN_OK;
}

int gdn_decode_step(const void* q, const void* k, const void* v, const float* alpha,
                    const float* beta, float* S_inout, void* out, int32_t batch,
                    int32_t heads, int32_t dk, int32_t dv, int32_t io_dtype,
                    gdn_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!q || !k || !v || !alpha || !beta || !S_inout || !out) return GDN_ERR_INVALID_ARG;
  if (batch < 1 || heads < 1) return GDN_ERR_INVALID_ARG;
  if (io_dtype != GDN_F32 && io_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if (dk != kDK || !supported_dv(dv)) return GDN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned4(alpha) || !aligned4(beta) ||
      !aligned16(S_inout) || !aligned16(out))
    return GDN_ERR_ALIGNMENT;
  const size_t es = io_dtype == GDN_BF16 ? 2 : 4;
  const size_t nh = (size_t)batch * heads;
  const Range r_out = span(out, nh * dv * es);
  const Range others[] = {span(q, nh * dk * es), span(k, nh * dk * es), span(v, nh * dv * es),
                          span(alpha, nh * 4), span(beta, nh * 4),
                          span(S_inout, nh * dv * dk * 4)};
  for (const Range& r : others)
    if (overlaps(r, r_out)) return GDN_ERR_INVALID_ARG;
  for (int i = 0; i < 5; ++i)
    if (overlaps(others[i], others[5])) return GDN_ERR_INVALID_ARG;
  const cudaError_t e =
      launch_decode_step(q, k, v, alpha, beta, S_inout, out, batch, heads, dv, io_dtype, stream);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_testing_prefill_prep(const void* q, const void* k, const void* v, const float* alpha,
                             const float* beta, const int32_t* cu_seqlens, int32_t batch,
                             int64_t seqlen, int32_t heads, void* images, size_t image_bytes,
                             gdn_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!q || !k || !v || !alpha || !beta || !images || batch < 1 || seqlen < 1 || heads < 1)
    return GDN_ERR_INVALID_ARG;
  const bool varlen = cu_seqlens != nullptr;
  const int64_t T_total = varlen ? seqlen : (int64_t)batch * seqlen;
  PrefillLaunch a{};
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.H = heads; a.dv = kDV;
  a.status = status_ptr();
  if (!a.status) return GDN_ERR_CUDA;
  a.map.cu_seqlens = cu_seqlens;
  a.map.N = batch;
  a.map.T = varlen ? T_total : seqlen;
  a.map.chunks_per_seq = varlen ? 0 : (seqlen + kC - 1) / kC;
  a.max_chunks = max_chunks_bound(batch, T_total, varlen, seqlen);
  if (image_bytes < (size_t)a.max_chunks * heads * prefill_tc_image_stride())
    return GDN_ERR_INVALID_ARG;
  void* offs = nullptr;
  if (varlen) {
    if (cudaMallocAsync(&offs, ((size_t)batch + 1) * 4, stream) != cudaSuccess) return GDN_ERR_CUDA;
    a.map.chunk_off = (int32_t*)offs;
    if (launch_chunk_offsets(cu_seqlens, batch, T_total, (int32_t*)offs, a.status, stream) !=
        cudaSuccess)
      return GDN_ERR_CUDA;
  }
  a.scratch = images;
  cudaError_t e = launch_prefill_tc(a, stream, /*prep_only=*/true);
  if (offs) cudaFreeAsync(offs, stream);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

size_t gdn_testing_prefill_image_stride(void) { return prefill_tc_image_stride(); }

int32_t gdn_testing_last_prefill_form(void) { return g_last_tc_form; }

void gdn_testing_set_trace(uint64_t* device_buf, int32_t max_chunks) {
  g_trace = device_buf;
  g_trace_chunks = device_buf ? (max_chunks < 256 ? max_chunks : 256) : 0;
}

int gdn_get_device_status(gdn_stream_t stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof v) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess) return GDN_ERR_CUDA;
  return (int)v;
}

uint64_t gdn_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char* gdn_prefill_path(int32_t io_dtype) {
  if (io_dtype == GDN_F32) return "simt-f32";
  if (io_dtype == GDN_BF16) return "tcgen05-bf16";
  return nullptr;
}

const char* gdn_version(void) { return "gdn-gb300 0.1.0 (sm_103a)"; }

const char* gdn_status_string(int s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported head geometry or dtype";
    case GDN_ERR_ALIGNMENT: return "pointer not aligned (16 B for tensors, 4 B for alpha/beta/cu_seqlens)";
    case GDN_ERR_CUDA: return "CUDA runtime error";
    case GDN_ERR_TIMEOUT: return "device: bounded wait timed out";
    case GDN_ERR_BAD_SEQLENS: return "device: malformed cu_seqlens";
    case GDN_ERR_SCRATCH_LIMIT: return "problem needs more than the 64 MiB static no-allocation scratch";
    default: return "unknown status";
  }
}

}  // extern "C"
