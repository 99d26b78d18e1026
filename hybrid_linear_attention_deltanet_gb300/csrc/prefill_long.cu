// Prefill of long sequences as a scan over segments of whole chunks, taken
// automatically by gdn_prefill for long sequences and on request by
// gdn_prefill_scan.
//
// Over the chunks of one sequence the state pass is affine in its start state
// (the recurrence of "Long-Context Aware Upcycling", Appendix A.3, Eq. 16-18):
// S_end = S_start A + B, where B is the end state from a zero start and A
// (dk x dk) the product of the segment's per-token transitions
// alpha_t (I - beta_t k_t k_t^T).  The chunked form walks the chunks of a
// sequence one after another (Appendix A.3, last paragraph), so one long
// sequence leaves most of the GPU idle.  Cut into P segments it runs as P
// chains joined by a short sequential scan over the segments' (A, B) pairs:
//   pass 1  every segment but the last, without outputs: the first from the
//           sequence's own start (-> B(0), its true end state), the middle
//           ones from zero (-> B) and, in the same launch, their A chains:
//           the same chunks from the identity with the inhomogeneous term U~
//           dropped (-> A);
//   scan    start(1) = B(0); start(j) = start(j-1) A(j-1) + B(j-1);
//   pass 2  every segment from its true start: the outputs, and the
//           sequence's final state from the last one.
// The critical path is two segments instead of P, and the chains without
// outputs load about two thirds of the bytes per chunk (neither Q^ nor P^;
// an A chain not even U~); the work is 3 - 3/P chains' worth.  Segments
// start on chunk boundaries of their sequence, so the per-chunk factors are
// the plain prefill's, computed once over the segmented packing (the same
// chunks in the same order).
//
// Which sequences are cut, and where, depends on nothing but the sequence's
// own length (or, for gdn_prefill_scan, the caller's segment count), so a
// sequence gives the same bits alone or packed with others.  A sequence left
// whole runs exactly the plain prefill's kernels on the same inputs.
#include <algorithm>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kScanRows = 16;   // state rows per scan CTA

// Segments of a sequence of n_c chunks: count P and chunks per segment.
// forced_P > 0: that many pieces (at most one per chunk); else the length
// rule.  An empty sequence is one empty segment.
__host__ __device__ __forceinline__ void seq_cut(int64_t n_c, int32_t forced_P, int64_t& P,
                                                 int64_t& seg) {
  int64_t p = 1;
  if (forced_P > 0) p = forced_P;
  else if (n_c >= kLongChunks) p = (n_c + kSegChunks - 1) / kSegChunks;
  if (n_c <= 1 || p <= 1) {
    P = 1;
    seg = n_c;
    return;
  }
  seg = (n_c + p - 1) / p;
  P = (n_c + seg - 1) / seg;
}

__device__ __forceinline__ int64_t seq_start(const int32_t* cu, int64_t T, int n) {
  return cu ? (int64_t)cu[n] : (int64_t)n * T;
}

// One CTA: each sequence's first segment slot, as the exclusive prefix
// seq_first[0..N] of the segment counts, after the cu_seqlens check of a
// packed batch (a malformed one flags GDN_ERR_BAD_SEQLENS and leaves an empty
// plan: no slot is used, nothing is written).
__global__ void __launch_bounds__(1024)
plan_counts_kernel(const int32_t* __restrict__ cu, int32_t N, int64_t T, int64_t T_total,
                   int32_t forced_P, int32_t* __restrict__ seq_first, unsigned* status) {
  __shared__ int bad;
  __shared__ int64_t carry;
  __shared__ int64_t warp_tot[32];
  if (threadIdx.x == 0) {
    bad = cu && (cu[0] != 0 || (int64_t)cu[N] != T_total) ? 1 : 0;
    carry = 0;
  }
  __syncthreads();
  if (cu)
    for (int n = threadIdx.x; n < N; n += blockDim.x)
      if (cu[n + 1] < cu[n]) bad = 1;
  __syncthreads();
  if (bad) {
    for (int n = threadIdx.x; n <= N; n += blockDim.x) seq_first[n] = 0;
    if (threadIdx.x == 0) flag_status(status, GDN_ERR_BAD_SEQLENS);
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = 0; base < N; base += blockDim.x) {
    const int n = base + threadIdx.x;
    int64_t c = 0;
    if (n < N) {
      const int64_t len = seq_start(cu, T, n + 1) - seq_start(cu, T, n);
      int64_t seg;
      seq_cut((len + kC - 1) / kC, forced_P, c, seg);
    }
    int64_t x = c;   // inclusive scan within the warp
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
      warp_tot[lane] = w;
    }
    __syncthreads();
    const int64_t before = carry + (warp ? warp_tot[warp - 1] : 0) + x - c;
    if (n < N) seq_first[n] = (int32_t)before;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = before + c;
    __syncthreads();
  }
  if (threadIdx.x == 0) seq_first[N] = (int32_t)carry;
}

// Thread i < N lays out sequence i's segments (token starts in the packing,
// sequence, role); thread i in [used, n_slots) marks slot i unused (an empty
// segment at the end of the packing).
__global__ void plan_segments_kernel(const int32_t* __restrict__ cu, int32_t N, int64_t T,
                                     int64_t T_total, int32_t forced_P,
                                     const int32_t* __restrict__ seq_first, int32_t n_slots,
                                     int32_t* __restrict__ seg_cu, int32_t* __restrict__ seg_seq,
                                     uint8_t* __restrict__ role) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int32_t used = seq_first[N];
  if (i < N) {
    const int n = (int)i;
    const int64_t s0 = seq_start(cu, T, n), len = seq_start(cu, T, n + 1) - s0;
    int64_t P, seg;
    seq_cut((len + kC - 1) / kC, forced_P, P, seg);
    const int32_t f = seq_first[n];
    for (int64_t j = 0; j < P && f + j < n_slots; ++j) {
      const int64_t s = f + j, a = s0 + j * seg * kC;
      seg_cu[s] = (int32_t)(a < s0 + len ? a : s0 + len);
      seg_seq[s] = n;
      role[s] = (j == 0 ? kSegFirst : 0) | (j == P - 1 ? kSegLast : 0);
    }
  }
  if (i >= used && i < n_slots) {
    seg_cu[i] = (int32_t)T_total;
    seg_seq[i] = -1;
    role[i] = kSegFirst | kSegLast;
  }
  if (i == 0) seg_cu[n_slots] = (int32_t)T_total;
}

// The scan, one CTA per (16 rows of the state, head) of a sequence: rows of S
// are independent under right-multiplication by A, so each CTA walks its
// sequence's segments on its own.  Thread c owns column c of its 16 rows;
// the previous start's rows sit in shared memory and column c of each A
// streams through registers in blocks of kScanBlk rows of A, the next block's loads
// (coalesced across the CTA) in flight while the current one is consumed:
// no A depends on the scan, so the stream never waits on the arithmetic.
constexpr int kScanBlk = 64;

__global__ void __launch_bounds__(256) seg_scan_kernel(float* __restrict__ S0seg,
                                                       const float* __restrict__ Bseg,
                                                       const float* __restrict__ Aseg,
                                                       const int32_t* __restrict__ seq_first,
                                                       int32_t N, int32_t H, int32_t dv) {
  __shared__ __align__(16) float prev[kScanRows][kDK];
  const int r0 = blockIdx.x * kScanRows, h = blockIdx.y, c = threadIdx.x;
  const int64_t st = (int64_t)dv * kDK;
  constexpr int kBlocks = kDK / kScanBlk;   // blocks of A rows per step
  for (int n = blockIdx.z; n < N; n += gridDim.z) {
    const int32_t f = seq_first[n], P = seq_first[n + 1] - f;
    if (P < 2) continue;   // the same for the whole CTA
    auto at = [&](const float* base, int j) { return base + ((int64_t)(f + j) * H + h) * st; };
    auto start_of = [&](int j) { return S0seg + ((int64_t)(f + j) * H + h) * st; };
    __syncthreads();   // the previous sequence is done with prev
    // start(1) = B(0): the first segment ran from the sequence's own start
#pragma unroll
    for (int r = 0; r < kScanRows; ++r) {
      const float x = at(Bseg, 0)[(r0 + r) * kDK + c];
      prev[r][c] = x;
      start_of(1)[(r0 + r) * kDK + c] = x;
    }
    // block t of the stream: step j = 2 + t / kBlocks, rows kScanBlk (t %
    // kBlocks) .. of A(j - 1)
    const int n_blk = (P - 2) * kBlocks;
    float a_cur[kScanBlk], a_nxt[kScanBlk], acc[kScanRows];
    auto load_blk = [&](int t, float* dst) {
      const float* A = at(Aseg, 1 + t / kBlocks) + (int64_t)(kScanBlk * (t % kBlocks)) * kDK + c;
#pragma unroll
      for (int i = 0; i < kScanBlk; ++i) dst[i] = A[(int64_t)i * kDK];
    };
    if (n_blk > 0) load_blk(0, a_cur);
    for (int t = 0; t < n_blk; ++t) {
      const int j = 2 + t / kBlocks, kb = t % kBlocks;
      if (t + 1 < n_blk) load_blk(t + 1, a_nxt);
      if (kb == 0) {
        const float* Bj = at(Bseg, j - 1);
#pragma unroll
        for (int r = 0; r < kScanRows; ++r) acc[r] = Bj[(r0 + r) * kDK + c];
        __syncthreads();   // prev holds start(j - 1)
      }
#pragma unroll
      for (int i = 0; i < kScanBlk; i += 4) {
#pragma unroll
        for (int r = 0; r < kScanRows; ++r) {
          const float4 p = *reinterpret_cast<const float4*>(&prev[r][kScanBlk * kb + i]);
          acc[r] = fmaf(p.x, a_cur[i], acc[r]);
          acc[r] = fmaf(p.y, a_cur[i + 1], acc[r]);
          acc[r] = fmaf(p.z, a_cur[i + 2], acc[r]);
          acc[r] = fmaf(p.w, a_cur[i + 3], acc[r]);
        }
      }
      if (kb == kBlocks - 1) {
        __syncthreads();   // every thread is done reading start(j - 1)
#pragma unroll
        for (int r = 0; r < kScanRows; ++r) {
          prev[r][c] = acc[r];
          start_of(j)[(r0 + r) * kDK + c] = acc[r];
        }
      }
#pragma unroll
      for (int i = 0; i < kScanBlk; ++i) a_cur[i] = a_nxt[i];
    }
  }
}

// The order in which a state pass's grid takes its units' x values: units
// that run, longest chain (most chunks) first, then those that do not run;
// ties in x order.  A grid larger than the SMs runs in waves, and a long
// chain started in a later wave would set the whole pass's length.  One CTA:
// the keys in shared memory, then each x counts the keys ahead of it.
constexpr int kMaxOrdered = 2048;

__global__ void __launch_bounds__(1024)
unit_order_kernel(SegRoute r, const int32_t* __restrict__ chunk_off, int32_t N, int32_t gx,
                  int32_t* __restrict__ order) {
  __shared__ int32_t key[kMaxOrdered];
  for (int x = threadIdx.x; x < gx; x += blockDim.x) {
    const UnitRoute u = route_unit(r, nullptr, nullptr, x, N, 0);
    const int s = x >= N ? x - N : x;
    key[x] = u.run ? chunk_off[s + 1] - chunk_off[s] : -1;
  }
  __syncthreads();
  for (int x = threadIdx.x; x < gx; x += blockDim.x) {
    const int32_t kx = key[x];
    int rank = 0;
    for (int y = 0; y < gx; ++y) rank += (key[y] > kx || (key[y] == kx && y < x)) ? 1 : 0;
    order[rank] = x;
  }
}

}  // namespace

bool long_form_applies(int64_t seqlen) {
  // dense: every sequence has seqlen tokens; packed: one may hold all of them
  return (seqlen + kC - 1) / kC >= kLongChunks;
}

LongPlan plan_long(int32_t N, int64_t seqlen, bool varlen, int32_t H, int32_t dv, int io_dtype,
                   int32_t forced_P) {
  LongPlan p;
  const int64_t T_total = varlen ? seqlen : (int64_t)N * seqlen;
  p.max_chunks = max_chunks_bound(N, T_total, varlen, seqlen);
  // a cut sequence of n_c chunks takes P - 1 < n_c / kSegChunks extra slots
  // (at most n_c - 1 when the count is forced)
  p.n_slots = forced_P > 0 ? std::min<int64_t>((int64_t)N * forced_P, N + p.max_chunks)
                           : N + p.max_chunks / kSegChunks + 1;
  const size_t slot_ints = align_up((size_t)(p.n_slots + 1) * 4, 256);
  const size_t states = align_up((size_t)p.n_slots * H * dv * kDK * 4, 256);
  const size_t work = io_dtype == GDN_BF16 ? prefill_tc_scratch_bytes(p.max_chunks, H, dv)
                                           : prefill_simt_scratch_bytes(p.max_chunks, H, dv);
  size_t o = 0;
  p.off_chunk_off = o; o += slot_ints;
  p.off_seg_cu = o;    o += slot_ints;
  p.off_seg_seq = o;   o += slot_ints;
  p.off_seq_first = o; o += align_up(((size_t)N + 1) * 4, 256);
  p.off_role = o;      o += align_up((size_t)p.n_slots, 256);
  p.off_order = o;     o += align_up((size_t)p.n_slots * 3 * 4, 256);
  p.off_work = o;      o += align_up(work, 256);
  p.off_S0seg = o;     o += states;
  p.off_Bseg = o;      o += states;
  p.off_Aseg = o;      o += states;
  p.bytes = o;
  return p;
}

cudaError_t launch_prefill_long(const PrefillLaunch& base, int io_dtype, const LongPlan& p,
                                int32_t forced_P, cudaStream_t stream) {
  const int32_t N = base.map.N, H = base.H, dv = base.dv;
  const bool varlen = base.map.cu_seqlens != nullptr;
  const int64_t T = varlen ? 0 : base.map.T;
  const int64_t T_total = varlen ? base.map.T : (int64_t)N * base.map.T;
  if (p.n_slots * 2 > 0x7fffffffLL || T_total > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int32_t slots = (int32_t)p.n_slots;
  char* scr = (char*)base.scratch;
  int32_t* chunk_off = (int32_t*)(scr + p.off_chunk_off);
  int32_t* seg_cu = (int32_t*)(scr + p.off_seg_cu);
  int32_t* seg_seq = (int32_t*)(scr + p.off_seg_seq);
  int32_t* seq_first = (int32_t*)(scr + p.off_seq_first);
  uint8_t* role = (uint8_t*)(scr + p.off_role);
  cudaError_t e;

  plan_counts_kernel<<<1, 1024, 0, stream>>>(base.map.cu_seqlens, N, T, T_total, forced_P,
                                             seq_first, base.status);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t threads = std::max<int64_t>(N, p.n_slots);
  plan_segments_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(
      base.map.cu_seqlens, N, T, T_total, forced_P, seq_first, slots, seg_cu, seg_seq, role);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_chunk_offsets(seg_cu, slots, T_total, chunk_off, base.status, stream)) !=
      cudaSuccess)
    return e;

  PrefillLaunch a = base;
  a.map.cu_seqlens = seg_cu;
  a.map.chunk_off = chunk_off;
  a.map.N = slots;
  a.map.T = T_total;
  a.map.chunks_per_seq = 0;
  a.max_chunks = p.max_chunks;   // the same chunks as the caller's packing
  a.scratch = scr + p.off_work;
  a.allow_overlap = false;
  a.state_dump = nullptr;
  a.S0 = nullptr;
  a.S_final = nullptr;
  a.route.seg_seq = seg_seq;
  a.route.role = role;
  a.route.S0 = base.S0;
  a.route.S_final = base.S_final;
  a.route.S0seg = (const float*)(scr + p.off_S0seg);
  a.route.Bseg = (float*)(scr + p.off_Bseg);
  a.route.Aseg = (float*)(scr + p.off_Aseg);
  if (a.cv.qkv) {
    a.cv.seg_seq = seg_seq;
    a.cv.seg_role = role;
  }
  int32_t* order = (int32_t*)(scr + p.off_order);
  auto run = [&](bool state_only, int pass) {
    a.state_only = state_only;
    a.route.pass = pass;
    a.route.order = nullptr;
    const int32_t gx = pass == 1 ? 2 * slots : slots;
    if (io_dtype == GDN_BF16 && gx <= kMaxOrdered) {
      int32_t* ord = order + (pass == 1 ? 0 : 2 * slots);
      unit_order_kernel<<<1, 1024, 0, stream>>>(a.route, chunk_off, slots, gx, ord);
      count_launches(1);
      const cudaError_t eo = cudaGetLastError();
      if (eo != cudaSuccess) return eo;
      a.route.order = ord;
    }
    return io_dtype == GDN_BF16 ? launch_prefill_tc(a, stream)
                                : launch_prefill_simt(a, io_dtype, stream);
  };
  // pass 1: the per-chunk factors, then every first and middle segment
  if ((e = run(false, 1)) != cudaSuccess) return e;
  // the scan: every later segment's true start
  seg_scan_kernel<<<dim3((unsigned)(dv / kScanRows), (unsigned)H,
                         (unsigned)std::min<int32_t>(N, 65535)),
                    256, 0, stream>>>((float*)(scr + p.off_S0seg), a.route.Bseg, a.route.Aseg,
                                      seq_first, N, H, dv);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // pass 2: every later segment from its true start, on the same factors
  return run(true, 2);
}

}  // namespace gdn
