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
// Arithmetic of the pre-recurrence steps ("Long-Context Aware Upcycling",
// Appendix A.3: the short convolution's SiLU and the q/k L2 norm), shared by
// gdn_prepare and by the tensor-core prep that runs the same steps on its
// tiles, so that the two give the same bits.
//
// F2: two fp32 values in one 64-bit register pair.  The .f32x2 forms of mul,
// add and fma (sm_100 onwards) round each half exactly as the scalar
// instruction does, at one issue for the pair.
struct F2 {
  uint64_t v;
};
__device__ __forceinline__ F2 f2(float lo, float hi) {
  F2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(F2 a, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
  F2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  F2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
  F2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}

// The special-function unit's base-2 exponential and reciprocal (a few ulp
// each; subnormal results flush to zero).
__device__ __forceinline__ float ex2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_sfu(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kNegLog2e = -1.44269504088896341f;
// SiLU x / (1 + e^-x), with e^-x = 2^(-x log2 e).  Far below zero e^-x
// overflows to inf and the reciprocal gives 0 (the limit); far above, it
// flushes to 0 and the result is x.  silu_pair gives the same bits per half.
__device__ __forceinline__ float silu_sfu(float x) {
  return __fmul_rn(x, rcp_sfu(__fadd_rn(ex2_sfu(__fmul_rn(x, kNegLog2e)), 1.f)));
}
__device__ __forceinline__ F2 silu_pair(F2 x) {
  float t0, t1, d0, d1;
  f2_split(f2_mul(x, f2(kNegLog2e, kNegLog2e)), t0, t1);
  f2_split(f2_add(f2(ex2_sfu(t0), ex2_sfu(t1)), f2(1.f, 1.f)), d0, d1);
  return f2_mul(x, f2(rcp_sfu(d0), rcp_sfu(d1)));
}
// A lane's part of a row's sum of squares over its 8 values y[0..7]: the
// even and the odd positions accumulate apart (in order), then add.
__device__ __forceinline__ float sumsq8(const float (&y)[8]) {
  float e = __fmul_rn(y[0], y[0]), o = __fmul_rn(y[1], y[1]);
#pragma unroll
  for (int k = 2; k < 8; k += 2) {
    e = fmaf(y[k], y[k], e);
    o = fmaf(y[k + 1], y[k + 1], o);
  }
  return __fadd_rn(e, o);
}
__device__ __forceinline__ float sumsq8(const F2 (&y)[4]) {
  F2 s = f2_mul(y[0], y[0]);
#pragma unroll
  for (int k = 1; k < 4; ++k) s = f2_fma(y[k], y[k], s);
  float e, o;
  f2_split(s, e, o);
  return __fadd_rn(e, o);
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
// Long sequences run as a scan over segments of whole chunks (prefill_long.cu):
// a sequence of at least kLongChunks chunks is cut into ceil(chunks /
// kSegChunks) pieces of equal length; shorter ones are one segment.
constexpr int64_t kLongChunks = 1024;
constexpr int64_t kSegChunks = 160;

// Role bits of a segment (one byte per segment slot).
constexpr uint8_t kSegFirst = 1, kSegLast = 2;

// Per-unit routing of the state pass over a segmented packing (the map's
// sequences are then segment slots).  pass 0: a plain call, every unit runs
// from S0 into S_final with outputs.  pass 1 (no outputs, except for a
// sequence left whole): the grid holds two units per slot and row block;
// x < N runs a sequence left whole from the caller's start into the caller's
// S_final with outputs, the first segment of a cut sequence from the
// caller's start into Bseg, a middle segment from zero into Bseg; x >= N runs
// the A chain of a middle segment into Aseg.  An A chain starts from the
// identity and drops U~: it carries the product A of the segment's
// transitions, S_end = S_start A + B, in its dk rows.  pass 2 (outputs):
// every segment of a cut sequence from its true start (the caller's S0 for
// the first, S0seg for the others; the last one's end into the caller's
// S_final).
struct SegRoute {
  int32_t pass = 0;
  const int32_t* seg_seq = nullptr;   // per slot: its sequence, -1 for an unused slot
  const uint8_t* role = nullptr;      // per slot: kSegFirst | kSegLast
  const float* S0 = nullptr;          // the caller's [N][H][dv][dk] starts, or nullptr (zero)
  float* S_final = nullptr;           // the caller's final states, or nullptr
  const float* S0seg = nullptr;       // [slots][H][dv][dk]
  float* Bseg = nullptr;
  float* Aseg = nullptr;              // [slots][H][dv][dk], rows 0 .. dk-1 used
  // (tensor-core path) the order in which the grid takes the units' x values
  // (longest chain first, units that do not run last), or nullptr: x order
  const int32_t* order = nullptr;
};

// Where one unit of the state pass starts and ends; S0 / S_final point at
// its sequence's (or slot's) [H][dv][dk] block.
struct UnitRoute {
  bool run, ident, write_out;   // ident: an A chain
  const float* S0;
  float* S_final;
};

__device__ __forceinline__ UnitRoute route_unit(const SegRoute& r, const float* S0,
                                                float* S_final, int x, int N, int64_t per_seq) {
  UnitRoute u{true, false, true, nullptr, nullptr};
  if (r.pass == 0) {
    u.S0 = S0 ? S0 + x * per_seq : nullptr;
    u.S_final = S_final ? S_final + x * per_seq : nullptr;
    return u;
  }
  const bool second = x >= N;
  const int s = second ? x - N : x;
  const int n = r.seg_seq[s];
  const uint8_t ro = r.role[s];
  const bool first = ro & kSegFirst, last = ro & kSegLast;
  u.run = n >= 0;
  if (r.pass == 1 && second) {          // A of a middle segment
    u.run = u.run && !first && !last;
    u.ident = true;
    u.write_out = false;
    u.S_final = r.Aseg + s * per_seq;
  } else if (r.pass == 1) {
    if (first && last) {                // a sequence left whole: the plain chain
      u.S0 = r.S0 ? r.S0 + n * per_seq : nullptr;
      u.S_final = r.S_final ? r.S_final + n * per_seq : nullptr;
    } else {                            // B of a first or middle segment
      u.run = u.run && !last;
      u.write_out = false;
      u.S0 = first && r.S0 ? r.S0 + n * per_seq : nullptr;
      u.S_final = r.Bseg + s * per_seq;
    }
  } else {                              // a segment of a cut sequence, with outputs
    u.run = u.run && !(first && last);
    u.S0 = !first ? r.S0seg + s * per_seq : r.S0 ? r.S0 + n * per_seq : nullptr;
    u.S_final = last && r.S_final ? r.S_final + n * per_seq : nullptr;
  }
  return u;
}

// Eq. 20's read-out applied by the tensor-core state pass to its outputs (the
// layer entry point): y = o / sqrt(mean(o^2) + eps) * w * act(gate) over the
// dv values of each (token, head), written over o.  Each 128-row unit of a
// head stores the per-row sums of squares of its half of o as it copies the
// rows out; the two units of a head run as a 2-CTA cluster, meet after their
// chains and then apply Eq. 20 to their halves (dv = 256 only).
struct NormGate {
  const __nv_bfloat16* gate = nullptr;   // [T_total, H, dv]; nullptr: plain outputs
  const float* w = nullptr;              // [dv]
  float eps = 0.f;
  int32_t act = 0;                       // GDN_GATE_SILU or GDN_GATE_SIGMOID
  float* part = nullptr;                 // scratch [T_total, H, 2]: the halves' sums of squares
                                         // (the split form's read-out)
  // fused form: one progress count per state unit (N * H * dv / 128, zeroed
  // by the caller): how many of the unit's chunks have their output rows
  // out, raised every few chunks; the per-chunk workers apply Eq. 20 to a
  // chunk's rows (sums of squares included) once both units of its head
  // have passed it.  nullptr: the two units of a head sum their halves as
  // they copy the rows out and finish the rows themselves after their
  // chains, as a 2-CTA cluster (the split form).
  uint32_t* flags = nullptr;
};

// The layer entry point's pre-recurrence steps, run by the tensor-core prep
// on its input tiles (Appendix A.3, the paragraph after Table 8 and the text
// under Eq. 16-21): the q, k, v tiles of a (chunk, head) come from the packed
// projection qkv and pass through the causal depthwise convolution of width 4
// and SiLU in shared memory (q and k then L2-normalised per head); alpha and
// beta come from a_raw / b_raw.  The processed keys also go to k_out, where
// the state pass reads its K tiles.  dv = 256 only.
struct ConvIn {
  const __nv_bfloat16* qkv = nullptr;        // [T_total, C], C = H (2 dk + dv); nullptr: off
  const float* conv_w = nullptr;             // [C, 4]
  const __nv_bfloat16* state_in = nullptr;   // [N, 3, C], or nullptr (zero history)
  __nv_bfloat16* state_out = nullptr;        // [N, 3, C], or nullptr
  const float* a_raw = nullptr;              // [T_total, H]
  const float* b_raw = nullptr;              // [T_total, H]
  const float* A_log = nullptr;              // [H]
  const float* dt_bias = nullptr;            // [H]
  __nv_bfloat16* k_out = nullptr;            // [T_total, H, dk]
  // over a segmented packing (the long-sequence form): each slot's sequence
  // and role, so that a segment's first rows continue its sequence's earlier
  // tokens and only a sequence's last segment writes state_out
  const int32_t* seg_seq = nullptr;
  const uint8_t* seg_role = nullptr;
};

// The backward's chunk-start states and state gradients dS' at dv = 256
// (bf16 I/O, where the tensor cores produce and consume them) sit in
// 4-column tiles: element (v, c) of a unit's [dv][dk] matrix at
// ((c / 4) * dv + v) * 4 + c % 4.  A warp whose lanes hold consecutive rows
// then stores contiguous bytes, and a GEMM that reads columns c .. c+3 of
// consecutive rows reads contiguous memory.  Both are bf16 there, as the
// forward's and the reverse pass's own MMAs read S and dS.  Other dv:
// row-major fp32.
__host__ __device__ constexpr bool tiled_states(int dv) { return dv == 256; }

// (the backward's forward re-run, split form) fp32 copies of per-chunk
// factors the tensor-core prep computes anyway, each [chunks * H][64][64]
// row-major with rows and columns past the chunk's valid rows zero: the raw
// Gram matrices K K^T and Q K^T, P^ = lower(Gam o Q K^T) / sqrt(dk),
// T = (I + A)^-1, T diag(beta gamma) and T diag(beta).  All null: none.
struct PrepSide {
  float* KK = nullptr;
  float* QK = nullptr;
  float* Ph = nullptr;
  float* Tm = nullptr;
  float* TmB = nullptr;
  float* TmU = nullptr;
};

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
  float* state_dump;    // tensor-core path: every chunk's start state, [chunks * H] units of
                        // dv x dk (bf16 in the tiled_states layout at dv = 256, the
                        // first half of the array; fp32 row-major otherwise), for the
                        // backward's forward re-run, or nullptr
  bool state_only;      // the per-chunk factors are already in scratch (an earlier call on
                        // the same inputs and map): run the state pass only
  SegRoute route;       // see SegRoute (pass != 0 forces the split form)
  NormGate ng;          // tensor-core path: see NormGate (forces the split form)
  ConvIn cv;            // tensor-core path: see ConvIn (q, k, v, alpha, beta unused)
  PrepSide side;        // tensor-core path, split form only: see PrepSide
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

// Long sequences as a scan over segments (prefill_long.cu).  The segmented
// form takes over a call when some sequence may have kLongChunks chunks
// (seqlen: T of a dense batch, T_total of a packed one) or when the caller
// fixes the segment count (forced_P > 0).  Its scratch: chunk offsets,
// token starts, sequences and roles of the segment slots, the path's
// per-chunk scratch over the caller's chunks, then three per-(slot, head)
// states (true starts, ends from zero, transition products A).
struct LongPlan {
  int64_t n_slots = 0, max_chunks = 0;
  size_t off_chunk_off = 0, off_seg_cu = 0, off_seg_seq = 0, off_seq_first = 0, off_role = 0,
         off_work = 0, off_S0seg = 0, off_Bseg = 0, off_Aseg = 0, off_order = 0, bytes = 0;
};
bool long_form_applies(int64_t seqlen);
LongPlan plan_long(int32_t N, int64_t seqlen, bool varlen, int32_t H, int32_t dv, int io_dtype,
                   int32_t forced_P);
// base: the caller's problem (map over its own sequences, S0 / S_final / out
// as given), scratch = the start of plan.bytes of device memory
cudaError_t launch_prefill_long(const PrefillLaunch& base, int io_dtype, const LongPlan& plan,
                                int32_t forced_P, cudaStream_t stream);

// The whole prefill (api.cu): which form a call takes, its scratch bytes,
// and its launches into scratch of that size (a: the caller's problem, with
// its status word; the form and layout as gdn_prefill_workspace_size states).
bool takes_long_form(int64_t seqlen, int32_t forced_P);
size_t prefill_scratch_bytes(int32_t batch, int64_t seqlen, int32_t heads, int32_t dv,
                             int32_t io_dtype, bool varlen, int32_t forced_P);
cudaError_t launch_prefill_any(PrefillLaunch a, int32_t io_dtype, int64_t seqlen,
                               int32_t forced_P, void* scratch, cudaStream_t stream);
// stream-ordered scratch from the library's pool
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t stream);
cudaError_t scratch_free(void* p, cudaStream_t stream);

// The backward's reverse state pass on the tensor cores (bf16 I/O): per
// (sequence, head, 128-row slice of dS), over the chunks in reverse, from
// dS_final (nullptr: zero) to dS0 (nullptr: not written); stores every
// chunk's end-state gradient dS' ([chunks * H] units of dv x dk: bf16 in the
// tiled_states layout at dv = 256, fp32 row-major otherwise) and dU
// ([chunks * H][64][dv] fp32).  images: the forward's per-chunk operand images over the
// same map; k, dout: the call's bf16 tensors.
struct ReverseLaunch {
  const void* k = nullptr;
  const void* dout = nullptr;
  SeqMap map{};
  int32_t H = 0, dv = 0;
  int64_t T_total = 0;
  const uint8_t* images = nullptr;
  const float* dS_final = nullptr;
  float* dS0 = nullptr;
  float* dSp = nullptr;
  float* dU = nullptr;
  unsigned* status = nullptr;
};
cudaError_t launch_reverse_tc(const ReverseLaunch& r, cudaStream_t stream);

cudaError_t launch_decode_step(const void* q, const void* k, const void* v, const float* alpha,
                               const float* beta, float* S, void* out, int32_t N, int32_t H,
                               int32_t dv, int io_dtype, cudaStream_t stream);

}  // namespace gdn
