// gdn_prefill_noalloc: the prefill for callers that must not allocate device
// memory during a call.
//
// gdn_prefill obtains its scratch (per-chunk operand images and, for packed
// batches, the chunk offsets) stream-ordered from a memory pool.  Some
// callers cannot allow that: serving loops that fix their memory footprint
// at start-up so that no request can fail on an allocation or fragment the
// pool mid-flight, hosts whose device memory is owned by another allocator
// that forbids raw CUDA allocations, and embedded runtimes with a static
// memory budget.  This entry point runs the same kernels with their scratch
// in one static device array, sized once and held by every GPU that loads
// the library until the process exits.
#include <mutex>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

// 64 MiB: room for 624 (chunk, head) units of 64 tokens on the bf16
// tensor-core path (about 6600 tokens of a 6-head layer) and about 450 on the
// fp32 path (about 4800 tokens).
constexpr size_t kNoAllocScratchBytes = 64ull << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of this device's static scratch.  Host code must not use
// the array's name as an address (it names a host-side stand-in), so the
// address is looked up once per device, with that device current.
void* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

bool is_aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return na && nb && a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" int gdn_prefill_noalloc(const void* q, const void* k, const void* v,
                                   const float* alpha, const float* beta, const float* S0,
                                   const int32_t* cu_seqlens, void* out, float* S_final,
                                   int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                                   int32_t dv, int32_t io_dtype, gdn_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (batch < 1 || seqlen < 0 || heads < 1) return GDN_ERR_INVALID_ARG;
  const bool varlen = cu_seqlens != nullptr;
  const int64_t T_total = varlen ? seqlen : (int64_t)batch * seqlen;
  if (T_total > 0 && (!q || !k || !v || !alpha || !beta || !out)) return GDN_ERR_INVALID_ARG;
  if (io_dtype != GDN_F32 && io_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if (dk != kDK || !supported_dv(dv)) return GDN_ERR_UNSUPPORTED;
  if (!is_aligned(q, 16) || !is_aligned(k, 16) || !is_aligned(v, 16) || !is_aligned(out, 16) ||
      !is_aligned(S0, 16) || !is_aligned(S_final, 16) || !is_aligned(alpha, 4) ||
      !is_aligned(beta, 4) || !is_aligned(cu_seqlens, 4))
    return GDN_ERR_ALIGNMENT;
  if (varlen && T_total > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  const size_t es = io_dtype == GDN_BF16 ? 2 : 4;
  const size_t ntok = (size_t)T_total * heads;
  const size_t state = (size_t)batch * heads * dv * dk * sizeof(float);
  const void* ins[] = {q, k, v, alpha, beta, S0, cu_seqlens};
  const size_t in_bytes[] = {ntok * dk * es, ntok * dk * es, ntok * dv * es, ntok * 4, ntok * 4,
                             S0 ? state : 0, varlen ? ((size_t)batch + 1) * 4 : 0};
  for (int i = 0; i < 7; ++i)
    if (ranges_overlap(ins[i], in_bytes[i], out, ntok * dv * es) ||
        ranges_overlap(ins[i], in_bytes[i], S_final, S_final ? state : 0))
      return GDN_ERR_INVALID_ARG;
  if (ranges_overlap(out, ntok * dv * es, S_final, S_final ? state : 0)) return GDN_ERR_INVALID_ARG;

  PrefillLaunch a{};
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.S0 = S0;
  a.out = out; a.S_final = S_final; a.H = heads;
  a.map.cu_seqlens = cu_seqlens;
  a.map.N = batch;
  a.map.T = varlen ? T_total : seqlen;
  a.map.chunks_per_seq = varlen ? 0 : (seqlen + kC - 1) / kC;
  a.max_chunks = max_chunks_bound(batch, T_total, varlen, seqlen);
  // bf16 I/O runs on the tensor cores, fp32 I/O on the CUDA cores; the same
  // launch forms as gdn_prefill (the fused cooperative one where it fits: its
  // ready flags are cleared before the launch, so the array's leftovers from
  // an earlier call do not matter)
  const bool tc = io_dtype == GDN_BF16;
  a.dv = dv;
  a.allow_overlap = true;
  const size_t off_bytes = varlen ? align_up(((size_t)batch + 1) * 4, 256) : 0;
  const size_t work_bytes = tc ? prefill_tc_scratch_bytes(a.max_chunks, heads, dv)
                               : prefill_simt_scratch_bytes(a.max_chunks, heads, dv);
  // a problem that may hold a sequence of kLongChunks chunks takes
  // gdn_prefill's segmented form, whose per-chunk factors alone (over 100 MB)
  // never fit here: rejected, so that both entry points always agree
  if (long_form_applies(seqlen) || off_bytes + work_bytes > kNoAllocScratchBytes)
    return GDN_ERR_SCRATCH_LIMIT;

  a.status = status_ptr();
  void* scratch = noalloc_scratch();
  if (!a.status || !scratch) return GDN_ERR_CUDA;
  a.scratch = (char*)scratch + off_bytes;
  cudaError_t e = cudaSuccess;
  if (varlen) {
    a.map.chunk_off = (int32_t*)scratch;
    e = launch_chunk_offsets(cu_seqlens, batch, T_total, (int32_t*)scratch, a.status, stream);
  }
  if (e == cudaSuccess) e = tc ? launch_prefill_tc(a, stream) : launch_prefill_simt(a, io_dtype, stream);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
