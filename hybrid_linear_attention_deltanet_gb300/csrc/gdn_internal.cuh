// Internal declarations shared by the library's translation units (never
// installed, never seen by callers).  Layouts and the meaning of every
// argument are those of include/gdn.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

// Head geometry implemented by the kernels (Table 8: head dim 256).  The
// value dimension dv is 256 (the configurations) or 512 (Table 8's value
// expansion dv = 2 dk); kDV is the 256 case.
constexpr int kDK = 256;
constexpr int kDV = 256;
constexpr int kDVMax = 512;
inline bool supported_dv(int32_t dv) { return dv == 256 || dv == 512; }
// Chunk length of the chunkwise-parallel form (Appendix A.3: C = 64).
constexpr int kC = 64;
// 1/sqrt(dk) for dk = 256: a power of two, so the scaling is exact.
constexpr float kScale = 0.0625f;

// ---------------------------------------------------------------------------
// element access for the two I/O types
__device__ __forceinline__ float ld_in(const float* p) { return *p; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// First device-side error wins; read back by gdn_get_device_status().
__device__ __forceinline__ void flag_status(unsigned* status, unsigned code) {
  if (status) atomicCAS(status, 0u, code);
}

// ---------------------------------------------------------------------------
// Chunk map.  Sequences are cut into chunks of kC tokens that restart at
// every sequence start; the last chunk of a sequence may be partial.  A dense
// batch is the packed case with cu[n] = n * T.
struct SeqMap {
  const int32_t* cu_seqlens;  // device, N+1 entries; nullptr for a dense batch
  const int32_t* chunk_off;   // device, N+1 exclusive prefix of chunk counts (varlen)
  int32_t N;                  // number of sequences
  int64_t T;                  // dense: tokens per sequence; varlen: T_total
  int64_t chunks_per_seq;     // dense only

  __device__ __forceinline__ int64_t seq_begin(int n) const {
    return cu_seqlens ? (int64_t)cu_seqlens[n] : (int64_t)n * T;
  }
  __device__ __forceinline__ int64_t seq_end(int n) const {
    return cu_seqlens ? (int64_t)cu_seqlens[n + 1] : (int64_t)(n + 1) * T;
  }
  __device__ __forceinline__ int64_t chunk_begin(int n) const {
    return cu_seqlens ? (int64_t)chunk_off[n] : (int64_t)n * chunks_per_seq;
  }
  __device__ __forceinline__ int64_t chunk_end(int n) const {
    return cu_seqlens ? (int64_t)chunk_off[n + 1] : (int64_t)(n + 1) * chunks_per_seq;
  }
  __device__ __forceinline__ int64_t total_chunks() const {
    return cu_seqlens ? (int64_t)chunk_off[N] : (int64_t)N * chunks_per_seq;
  }
  // Global chunk ci -> (sequence n, first token t0, valid rows L).  False when
  // ci is past the last chunk (grids are sized by a host-side upper bound).
  __device__ __forceinline__ bool locate(int64_t ci, int& n, int64_t& t0, int& L) const {
    if (ci >= total_chunks()) return false;
    if (cu_seqlens) {
      int lo = 0, hi = N - 1;  // last n with chunk_off[n] <= ci
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)chunk_off[mid] <= ci) lo = mid; else hi = mid - 1;
      }
      n = lo;
    } else {
      n = (int)(ci / chunks_per_seq);
    }
    t0 = seq_begin(n) + (ci - chunk_begin(n)) * kC;
    const int64_t rem = seq_end(n) - t0;
    L = rem < kC ? (int)rem : kC;
    return true;
  }
};

// Upper bound on the number of chunks: sum_n ceil(len_n / C) <= (T_total + N (C-1)) / C.
inline int64_t max_chunks_bound(int32_t N, int64_t T_total, bool varlen, int64_t T_dense) {
  if (!varlen) return (int64_t)N * ((T_dense + kC - 1) / kC);
  return (T_total + (int64_t)N * (kC - 1)) / kC;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// host-side count of kernel launches (gdn_kernel_launches)
void count_launches(int n);

// device address of the current device's status word (nullptr on failure)
unsigned* status_ptr();

// ---------------------------------------------------------------------------
// launchers (one translation unit each)
struct PrefillLaunch {
  const void* q; const void* k; const void* v;
  const float* alpha; const float* beta; const float* S0;
  void* out; float* S_final;
  SeqMap map;
  int32_t H;
  int32_t dv;           // 256 or 512
  int64_t max_chunks;   // grid bound for per-chunk kernels
  unsigned* status;
  void* scratch;        // device scratch of the size the path's *_scratch_bytes asks for
  bool allow_overlap;   // tensor-core path may run prep and state pass in one cooperative launch
  float* state_dump;    // tensor-core path: every chunk's start state, [chunks * H][dv][dk]
                        // fp32 (the backward's forward re-run), or nullptr
  bool state_only;      // tensor-core path: the per-chunk images are already in scratch
                        // (an earlier call on the same inputs and map); run the state pass only
};

cudaError_t launch_chunk_offsets(const int32_t* cu_seqlens, int32_t N, int64_t T_total,
                                 int32_t* chunk_off, unsigned* status, cudaStream_t stream);

// CUDA-core (fp32 FFMA) chunkwise path: used for fp32 I/O.
size_t prefill_simt_scratch_bytes(int64_t max_chunks, int32_t H, int32_t dv);
cudaError_t launch_prefill_simt(const PrefillLaunch& a, int io_dtype, cudaStream_t stream);

// Tensor-core (tcgen05) chunkwise path: used for bf16 I/O.
size_t prefill_tc_scratch_bytes(int64_t max_chunks, int32_t H, int32_t dv);
cudaError_t launch_prefill_tc(const PrefillLaunch& a, cudaStream_t stream, bool prep_only = false);
size_t prefill_tc_image_stride();
// phase-timeline buffer of the tensor-core state pass (test hook)
extern uint64_t* g_trace;
extern int32_t g_trace_chunks;
// launch form of the last tensor-core prefill on this process: 1 fused, 0 split
extern int32_t g_last_tc_form;

cudaError_t launch_decode_step(const void* q, const void* k, const void* v, const float* alpha,
                               const float* beta, float* S, void* out, int32_t N, int32_t H,
                               int32_t dv, int io_dtype, cudaStream_t stream);

}  // namespace gdn
