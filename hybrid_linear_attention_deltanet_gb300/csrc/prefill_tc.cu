// Chunkwise prefill on the 5th-generation tensor cores (tcgen05, bf16
// operands, fp32 accumulation in TMEM, fp32 master state).  Used for bf16 I/O.
//
// Chunked form of the gated delta rule (Appendix A.3 of "Long-Context Aware
// Upcycling": chunks of C = 64 tokens, intra-chunk delta corrections batched
// through the WY representation, state carried across chunks sequentially).
// For a chunk with start state S (dv x dk), rows r, j < L, G = cumsum(log
// alpha), gamma = exp(G), Gam_rj = exp(G_r - G_j), d_r = gamma_L / gamma_r:
//   A  = strict_lower(beta_r Gam_rj k_r.k_j),   T = (I + A)^{-1}
//   W  = T diag(beta gamma) K,  U~ = T diag(beta) V,  P^ = lower(Gam Q K^T)/sqrt(dk)
//   Q^ = diag(gamma) Q / sqrt(dk)
//   U  = U~ - W S^T,  O = Q^ S^T + P^ U,  S' = gamma_L S + (diag(d) U)^T K
//
// Prep (fully parallel over (chunk, head) items):
//   TMA tensor copies of the K, Q, V tiles; [K;Q] K^T on tcgen05 (M=128, N=64,
//   K=256) -> A and P^; T by a two-level recursive block inverse in fp32 on
//   the CUDA cores; W^T = K^T T_w^T and U~^T = V^T T_u^T on tcgen05.  W, Q^,
//   U~^T and the decay factors are laid out in shared memory as ready-to-load
//   swizzled operand images and written to scratch by TMA bulk stores.
// State pass (one unit per (sequence, head, 128-row half of S)):
//   rows of S are independent, so each unit owns 128 rows (the MMA M).  The
//   bf16 copy of its S rows lives in TMEM as an A operand; the fp32 master
//   copy lives in registers.  Per chunk: [D_U | D_O] = S [W | Q^]^T (M=128,
//   N=128, K=256, A from TMEM); U = U~ - D_U and d*U -> bf16, stored back
//   into TMEM as A operands; D_S = (dU)^T K (N=256, K=64, K straight from the
//   input by a TMA tensor copy) and D_O += U^T P^^T; S = gamma_L S + D_S;
//   O -> out.  W, Q^, K and P^ are double-buffered (two chunks ahead).
//
// Two launch forms:
//   fused  one cooperative launch, one CTA per SM.  The first CTAs run the
//          state units; the others are prep workers that take items in
//          chunk-position order and publish each finished image with a
//          release flag, which a state unit acquires before it copies that
//          chunk's images.  The sequential pass starts after the first
//          chunk position instead of after the whole prep.  Used when the
//          state units leave enough SMs over for the workers.
//   split  a persistent prep kernel over all items (two CTAs per SM), then
//          the state kernel (one CTA per unit).
//
// Shared-memory operand images use the 128-byte swizzle: rows of 64 bf16,
// 16-byte chunk index XOR (row % 8), 8-row groups 1024 bytes apart.
//   K-major image of an R x K operand: K blocks of 64 columns, R*128 bytes apart.
//   MN-major image: one 128-byte row per K index holding 64 MN elements;
//   64-element MN blocks LBO bytes apart.
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

using namespace sm100;

// ---- scratch image per (chunk, head)
// [W | Q^] as one N = 128 MN-major B operand of 256 K-rows (c): 64-row
// blocks interleaved, W_0 Q^_0 W_1 Q^_1 W_2 Q^_2 W_3 Q^_3 (8 KB each), where
// W_b / Q^_b hold the 128-byte rows c in [64b, 64b + 64) = W[0..63][c] /
// Q^[0..63][c] (the layout of the per-chunk kernel's K/Q tile buffer)
constexpr size_t kImgWQ = 0;
constexpr size_t kImgP = 65536;       // P^  : K-major B image, 64 rows x 64
// per 128-row half h of S: U~^T rows [128h, 128h+128) (128-byte swizzled,
// 16 KB) followed by the chunk's decay block (512 B: d_r = gamma_L / gamma_r
// for r < L else 0, then G_r), so that one bulk copy brings both
constexpr size_t kImgU0 = 73728;
constexpr size_t kImgHalf = 16896;    // 16384 + 512
constexpr size_t kImgDecay = 16384;   // offset of the decay block inside a half
constexpr size_t kImgStride = 107520; // kImgU0 + 2 * kImgHalf (dv = 256), a multiple of 1 KB
// At dv = 512 the image carries four 128-row slices of U~^T, each with its
// decay block: kImgU0 + 4 * kImgHalf = 141312 bytes (also a multiple of 1 KB).
__host__ __device__ constexpr size_t img_stride(int dv) {
  return kImgU0 + (size_t)(dv / 128) * kImgHalf;
}
static_assert(img_stride(256) == kImgStride && img_stride(512) % 1024 == 0, "image strides");

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&t);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// exp(x) = 2^(x log2 e) on the special-function unit; results below the
// smallest normal float flush to zero (they only scale terms that are
// already negligible)
__device__ __forceinline__ float exp_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
  return y;
}

// byte offset of 16-byte chunk `ch` (0..7) of row `row` in a 128-byte-swizzled image
__device__ __forceinline__ uint32_t sw_chunk(uint32_t row, uint32_t ch) {
  return row * 128u + ((ch ^ (row & 7u)) << 4);
}

// Bounded wait for a ready flag (fused form): give up after one second.
constexpr uint64_t kReadyWaitNs = 1000000000ull;
// (fused form with the read-out) a state unit reports its output progress
// every kReadoutStep chunks
constexpr int kReadoutStep = 16;

// ============================================================ prep
constexpr int kPrepThreads = 256;
// row stride (floats) of the fp32 64 x 64 tiles: rows stay 16-byte aligned,
// so the block inverse reads four consecutive elements of a row at once
constexpr int kLd = 68;
constexpr int kPrepTraceOffset = 4096;   // uint64 slots before the prep timeline
// global-timer timeline of one call (test hook): per state unit u < 128 its
// start, first chunk top and end; per prep worker w < 200 its start and end;
// the start of each of the first 240 items of worker 0
constexpr int kUnitTimes = 3072, kMaxTracedUnits = 128;
constexpr int kWorkerTimes = kUnitTimes + 3 * kMaxTracedUnits, kMaxTracedWorkers = 200;
constexpr int kItemTimes = kWorkerTimes + 2 * kMaxTracedWorkers, kMaxTracedItems = 240;
static_assert(kItemTimes + kMaxTracedItems <= kPrepTraceOffset, "trace layout");
constexpr int kPrepIO = 64;              // thread that issues the prep's bulk copies

// Shared-memory layout of the prep (offsets from the 1024-aligned base).
// K/Q buffers of 64 KB (two in the fused form); K-block b at b*16K holds
// rows 0-63 of K, then rows 64-127 of Q.  Within a buffer's life the Q slots
// hold Q, then the Q^ rows; after the W / U~ MMAs the K slots hold the W
// rows, so that the buffer is the [W | Q^] image.  Split form: Q^ leaves
// early, V lands in the Q slots and the U~^T rows go there after the MMAs.
// Fused form: V (four 64-column blocks of 8 KB) has a buffer of its own,
// which afterwards holds the two halves of U~^T with their decay blocks in
// image layout, and P^ is staged too: an item leaves in three bulk stores.
template <bool kFused>
struct PrepSmem {
  static constexpr uint32_t KQ = 0;
  static constexpr uint32_t V = 65536u * (kFused ? 2 : 1);
  static_assert(!kFused || 2 * kImgHalf <= 34816, "U~^T halves fit the V buffer");
  static constexpr uint32_t PS = V + (kFused ? 34816u : 0u);   // V: 2 x 16896 rounded to 1 KB
  static constexpr uint32_t A = PS + (kFused ? 8192u : 0u);   // fp32 [64][kLd]; then T_w, T_u
  static constexpr uint32_t TW = A;                  //   (bf16 K-major 64 x 64, 8 KB each)
  static constexpr uint32_t TU = A + 8192;
  static constexpr uint32_t T = A + 64 * kLd * 4;    // fp32 [64][kLd]
  static constexpr uint32_t Y1 = T + 64 * kLd * 4;   // fp32 [2][16][16]; decay block at the end
  static constexpr uint32_t Y2 = Y1 + 2 * 256 * 4;   // fp32 [32][33]
  static constexpr uint32_t G = Y2 + 32 * 33 * 4;    // fp32 [64]
  static constexpr uint32_t B = G + 256;             // fp32 [64]
  static constexpr uint32_t GAM = B + 256;           // fp32 [64]: gamma_r = exp(G_r)
  static constexpr uint32_t END = GAM + 256;
  static constexpr uint32_t BYTES = END + 1024;      // + alignment slack
};

struct PrepItem {
  int64_t ci = 0, t0 = 0;   // global chunk index, first token
  int h = 0, L = 0;         // head, valid rows
  int n = 0;                // sequence
};


// Item j of the prep.  kOrdered: chunk positions in order (position p of
// every sequence and head before position p + 1), so that the next chunk of
// every state unit is among the first finished; otherwise global chunk order
// with the head fastest.  False for positions past a sequence's end.
template <bool kOrdered>
__device__ __forceinline__ bool prep_item(const SeqMap& map, int32_t H, int64_t j, PrepItem& it) {
  if (!kOrdered) {
    it.ci = j / H;
    it.h = (int)(j % H);
    return map.locate(it.ci, it.n, it.t0, it.L);
  }
  const int64_t nh = (int64_t)map.N * H;
  const int64_t p = j / nh;
  const int rem = (int)(j - p * nh);
  const int n = rem / H;
  it.n = n;
  it.h = rem - n * H;
  const int64_t cb = map.chunk_begin(n);
  if (cb + p >= map.chunk_end(n)) return false;
  it.ci = cb + p;
  it.t0 = map.seq_begin(n) + p * kC;
  const int64_t left = map.seq_end(n) - it.t0;
  it.L = left < kC ? (int)left : kC;
  return true;
}

// The prep over items worker, worker + n_workers, ... < n_items.
// kFused: two K/Q buffers (the next item's tiles load during this one),
// items in chunk-position order, and a ready flag per finished item.
// kSide: also the PrepSide copies (split form).
template <bool kFused, bool kSide = false>
__device__ __forceinline__ void prep_role(uint8_t* sm, const CUtensorMap* tm_q,
                                          const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                          const float* __restrict__ alpha,
                                          const float* __restrict__ beta, const SeqMap& map,
                                          int32_t H, uint8_t* __restrict__ scratch,
                                          uint32_t* ready, unsigned* status, int32_t dv,
                                          const ConvIn& cv, uint64_t* __restrict__ trace,
                                          uint64_t* __restrict__ timeline, int64_t n_items,
                                          int64_t worker, int64_t n_workers,
                                          const PrepSide& side = PrepSide{}) {
  constexpr int kBufs = kFused ? 2 : 1;
  using Lay = PrepSmem<kFused>;
  float* sA = (float*)(sm + Lay::A);
  float* sT = (float*)(sm + Lay::T);
  float* sY1 = (float*)(sm + Lay::Y1);
  float* sY2 = (float*)(sm + Lay::Y2);
  float* sG = (float*)(sm + Lay::G);
  float* sB = (float*)(sm + Lay::B);
  float* sGam = (float*)(sm + Lay::GAM);
  float* sDecay = (float*)(sm + Lay::Y1);   // d[64], G[64] staged for the bulk store
  __shared__ uint64_t bar_kq[kBufs], bar_v, bar_a, bar_bc;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, hv = warp >> 2;
  const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
  // optional phase timeline (test hook): thread 0 of worker 0 stamps its SM
  // cycle counter at 9 points of its item kTracedItem, and the bulk-copy
  // thread at 8 points around its copy issues
  constexpr int kTracedItem = 4;
  bool tracing = false;
  auto stamp = [&](int k) {
    if (tracing && tid == 0) trace[k] = clock64();
  };
  auto io_stamp = [&](int k) {
    if (tracing && tid == kPrepIO) trace[9 + k] = clock64();
  };
  const bool timed = timeline && tid == 0 && worker < kMaxTracedWorkers;
  if (timed) timeline[kWorkerTimes + 2 * worker] = globaltimer_ns();
  int n_done = 0;

  if (tid == 0) {
    for (int b = 0; b < kBufs; ++b) mbar_init(&bar_kq[b], 1);
    mbar_init(&bar_v, 1);
    mbar_init(&bar_a, 1);
    mbar_init(&bar_bc, 1);
    fence_barrier_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  auto next_valid = [&](int64_t j, PrepItem& it) -> int64_t {
    for (; j < n_items; j += n_workers)
      if (prep_item<kFused>(map, H, j, it)) return j;
    return n_items;
  };
  // copies issued by kPrepIO, counted per barrier for a clean exit after a timeout
  uint32_t n_kq[kBufs] = {}, n_v = 0;
  // (conv) q, k and v heads are heads h, H + h and 2H + h of the packed qkv rows
  const bool conv = cv.qkv != nullptr;
  const int kh0 = conv ? H : 0, vh0 = conv ? 2 * H : 0;
  auto issue_kq = [&](const PrepItem& it, int b) {
    uint8_t* dst = sm + Lay::KQ + b * 65536;
    mbar_arrive_expect_tx(&bar_kq[b], 65536);
    for (int kb = 0; kb < 4; ++kb) {
      tma_load_3d(dst + kb * 16384, tm_k, kb * 64, kh0 + it.h, (int32_t)it.t0, &bar_kq[b]);
      tma_load_3d(dst + kb * 16384 + 8192, tm_q, kb * 64, it.h, (int32_t)it.t0, &bar_kq[b]);
    }
    ++n_kq[b];
  };
  // V columns [256 vh, 256 vh + 256) of the item
  auto issue_v = [&](const PrepItem& it, int vh, uint8_t* dst, uint32_t block_stride) {
    mbar_arrive_expect_tx(&bar_v, 32768);
    for (int b = 0; b < 4; ++b)
      tma_load_3d(dst + b * block_stride, tm_v, kDK * vh + b * 64, vh0 + it.h, (int32_t)it.t0,
                  &bar_v);
    ++n_v;
  };
  auto img_of = [&](const PrepItem& it) {
    return scratch + (size_t)(it.ci * H + it.h) * img_stride(dv);
  };
  // (kPrepIO) the item's bulk stores have landed: raise its ready flag
  auto publish = [&](const PrepItem& it) {
    bulk_wait_all();
    fence_proxy_async_global();
    st_release_gpu(ready + it.ci * H + it.h, 1u);
  };

  // alpha and beta of token t0 + tid of an item: read, or (conv) computed
  // from the gate projections as the separate pre-recurrence pass does
  auto gates_of = [&](const PrepItem& it, float& a, float& b) {
    const int64_t idx = (it.t0 + tid) * H + it.h;
    if (conv) {
      const float x = __ldg(cv.a_raw + idx) + __ldg(cv.dt_bias + it.h);
      const float sp = x > 20.f ? x : log1pf(expf(x));
      a = expf(-expf(__ldg(cv.A_log + it.h)) * sp);
      b = 1.f / (1.f + expf(-__ldg(cv.b_raw + idx)));
    } else {
      a = alpha[idx];
      b = beta[idx];
    }
  };
  // (conv) the width-4 causal convolution + SiLU (and the L2 norm for q, k)
  // of one 64 x 256 tile in place: warp w takes rows 8w .. 8w+7, lane l its
  // 8 channels.  The taps and the inputs before the chunk (the sequence's
  // earlier tokens, its carried state or zeros) load before the wait for the
  // tile's copy; then every warp reads its eight rows and the three before
  // them, all warps meet, and each row's arithmetic (the separate pass's,
  // value for value) runs independently of the others.  Keys (rows < L) also
  // go to k_out; the item holding a sequence's last token writes the
  // sequence's last three inputs to state_out.
  auto conv_tile = [&](const PrepItem& it, uint8_t* base, uint32_t blk_stride, int64_t ch0,
                       bool l2, bool keys, uint64_t* bar, uint32_t parity) {
    const int64_t C = (int64_t)3 * H * kDK;
    const int r0 = 8 * warp;
    const int64_t ch = ch0 + 8 * lane;
    uint8_t* blk = base + (lane >> 3) * blk_stride;
    const uint32_t cb = lane & 7;
    auto cell = [&](int r) { return reinterpret_cast<uint4*>(blk + r * 128 + ((cb ^ (r & 7)) << 4)); };
    // element k of 8 packed bf16 values
    auto elt = [](const uint4& u, int k) {
      const uint32_t v = k < 2 ? u.x : k < 4 ? u.y : k < 6 ? u.z : u.w;
      return (k & 1) ? bf16_hi(v) : bf16_lo(v);
    };
    float w[4][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 t = __ldg(reinterpret_cast<const float4*>(cv.conv_w + (ch + i) * 4));
      w[0][i] = t.x; w[1][i] = t.y; w[2][i] = t.z; w[3][i] = t.w;
    }
    const int64_t sb = map.seq_begin(it.n), se = map.seq_end(it.n);
    int64_t nseq = it.n;
    bool seq_first = true, seq_last = true;
    if (cv.seg_seq) {   // it.n is a segment slot
      nseq = cv.seg_seq[it.n];
      seq_first = (cv.seg_role[it.n] & kSegFirst) != 0;
      seq_last = (cv.seg_role[it.n] & kSegLast) != 0;
    }
    // the three inputs before row r0 (packed bf16): the chunk's earlier
    // tokens (warp 0: from global memory, loaded before the copy lands) or
    // the tile's rows, read before any warp replaces them
    uint4 hist[3];
    if (r0 == 0) {
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int64_t t = it.t0 - 3 + j;
        if (t >= sb || !seq_first)
          hist[j] = __ldg(reinterpret_cast<const uint4*>(cv.qkv + t * C + ch));
        else if (cv.state_in)
          hist[j] = __ldg(reinterpret_cast<const uint4*>(cv.state_in + (nseq * 3 + (t - sb + 3)) * C + ch));
        else
          hist[j] = make_uint4(0, 0, 0, 0);
      }
    }
    if (!mbar_wait(bar, parity)) s_abort = 1;
    if (r0 > 0) {
#pragma unroll
      for (int j = 0; j < 3; ++j) hist[j] = *cell(r0 - 3 + j);
    }
    __syncthreads();   // every window is in registers before rows are replaced
    const bool last_chunk = it.t0 + it.L == se && seq_last;
    // two rows at a time (this warp's own rows, read before it replaces
    // them): their arithmetic and their reductions interleave
#pragma unroll 1
    for (int i = 0; i < 8; i += 2) {
      const uint4 in[5] = {hist[0], hist[1], hist[2], *cell(r0 + i), *cell(r0 + i + 1)};
      // gdn_prepare's arithmetic, one channel at a time (the same bits)
      float y[2][8], ss[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float acc = __fmul_rn(w[0][k], elt(in[u], k));
          acc = fmaf(w[1][k], elt(in[u + 1], k), acc);
          acc = fmaf(w[2][k], elt(in[u + 2], k), acc);
          acc = fmaf(w[3][k], elt(in[u + 3], k), acc);
          y[u][k] = silu_sfu(acc);
        }
        ss[u] = sumsq8(y[u]);
      }
      if (l2) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          ss[0] += __shfl_xor_sync(0xffffffffu, ss[0], o);
          ss[1] += __shfl_xor_sync(0xffffffffu, ss[1], o);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float rr = rsqrtf(ss[u] + 1e-6f);
#pragma unroll
          for (int k = 0; k < 8; ++k) y[u][k] *= rr;
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint4 pk;
        pk.x = pack_bf16(y[u][0], y[u][1]);
        pk.y = pack_bf16(y[u][2], y[u][3]);
        pk.z = pack_bf16(y[u][4], y[u][5]);
        pk.w = pack_bf16(y[u][6], y[u][7]);
        const int r = r0 + i + u;
        *cell(r) = pk;
        if (keys && r < it.L)
          *reinterpret_cast<uint4*>(cv.k_out + ((it.t0 + r) * H + it.h) * kDK + 8 * lane) = pk;
        if (cv.state_out && last_chunk && r == it.L - 1) {
#pragma unroll
          for (int j = 0; j < 3; ++j)
            *reinterpret_cast<uint4*>(cv.state_out + (nseq * 3 + j) * C + ch) = in[u + 1 + j];
        }
      }
      hist[0] = in[2];
      hist[1] = in[3];
      hist[2] = in[4];
    }  };

  PrepItem cur, nxt, prev;
  bool have_prev = false;
  int64_t j = next_valid(worker, cur);
  uint32_t kq_ph[kBufs] = {};   // parity of each K/Q buffer's next phase
  uint32_t ph = 0;              // parity of bar_a for this item
  uint32_t vph = 0, bcph = 0;   // parities of bar_v / bar_bc (dv / 256 uses per item)
  int buf = 0;
  float a_cur = 1.f, b_cur = 0.f;   // this item's gates (threads < C)
  if (kFused && j < n_items) {
    if (tid == kPrepIO) {
      issue_kq(cur, 0);
      issue_v(cur, 0, sm + Lay::V, 8192);
    }
    if (tid < kC && tid < cur.L) gates_of(cur, a_cur, b_cur);
  }

  while (j < n_items) {
    const int64_t jn = next_valid(j + n_workers, nxt);
    const int L = cur.L;
    uint8_t* const img = img_of(cur);
    uint8_t* const kq = sm + Lay::KQ + buf * 65536;
    tracing = trace && worker == 0 && n_done == kTracedItem;
    stamp(0);
    if (timed && worker == 0 && n_done < kMaxTracedItems) timeline[kItemTimes + n_done] = globaltimer_ns();
    ++n_done;
    float a_nx = 1.f, b_nx = 0.f;
    if (!kFused) {
      // one buffer: the previous item's stores must have read it
      if (tid == kPrepIO) {
        bulk_wait_read_all();
        issue_kq(cur, 0);
      }
      if (tid < kC && tid < L) gates_of(cur, a_cur, b_cur);
    } else if (jn < n_items && tid < kC && tid < nxt.L) {   // gates of the next item
      gates_of(nxt, a_nx, b_nx);
    }
    // decay prefix G_r = sum_{s <= r} log alpha_s (pad rows: log alpha = 0, beta = 0)
    float g_scan = 0.f;
    if (tid < kC) {
      const bool ok = tid < L;
      g_scan = ok ? logf(a_cur) : 0.f;
      sB[tid] = ok ? b_cur : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, g_scan, o);
        if (lane >= o) g_scan += y;
      }
      if (tid < 32) sG[tid] = g_scan;
    }
    for (int e = tid; e < 64 * kLd; e += kPrepThreads) sT[e] = 0.f;
    __syncthreads();
    if (tid >= 32 && tid < kC) sG[tid] = g_scan + sG[31];
    if (tid < kC) sGam[tid] = exp_fast(tid < 32 ? g_scan : g_scan + sG[31]);
    __syncthreads();
    stamp(1);

    if (conv) {   // k, q: convolution + SiLU + L2 in place, once the tiles are in
      conv_tile(cur, kq, 16384, (int64_t)(H + cur.h) * kDK, true, true, &bar_kq[buf], kq_ph[buf]);
      conv_tile(cur, kq + 8192, 16384, (int64_t)cur.h * kDK, true, false, &bar_kq[buf],
                kq_ph[buf]);
      fence_proxy_async_smem();
      __syncthreads();
    }
    // ---- [K; Q] K^T  ->  TMEM columns [0, 64): lanes 0-63 K K^T, 64-127 Q K^T
    if (tid == 0) {
      if (!mbar_wait(&bar_kq[buf], kq_ph[buf])) {
        s_abort = 1;
      } else {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(128, 64, 0, 0);
        const uint32_t base = smem_u32(kq);
        for (int s = 0; s < 16; ++s) {
          const uint64_t d = smem_desc(base + (s >> 2) * 16384u + (s & 3) * 32u, 16, 1024,
                                       kSwizzle128B);
          mma_bf16(tmem, d, d, idesc, s > 0);
        }
        mma_commit(&bar_a);
      }
    }
    // Q^ = gamma_r Q / sqrt(dk) in registers, row c of its MN-major image
    // (Q^[0..63][c]), so that it sits beside W as one N = 128 operand
    uint32_t qv[8][4];
    if (!mbar_wait(&bar_kq[buf], kq_ph[buf])) s_abort = 1;
    {
      const int c = tid;   // d_k column, 0..255
      const uint8_t* qb = kq + (c >> 6) * 16384 + 8192;
      const uint32_t cc = c & 63;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r0 = 8 * ch + 2 * e, r1 = r0 + 1;
          const float q0 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
              qb + r0 * 128 + ((((cc >> 3) ^ (r0 & 7)) << 4) | ((cc & 7) << 1))));
          const float q1 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
              qb + r1 * 128 + ((((cc >> 3) ^ (r1 & 7)) << 4) | ((cc & 7) << 1))));
          const float g0 = r0 < L ? kScale * sGam[r0] : 0.f;
          const float g1 = r1 < L ? kScale * sGam[r1] : 0.f;
          qv[ch][e] = pack_bf16(q0 * g0, q1 * g1);
        }
      }
    }
    kq_ph[buf] ^= 1u;
    stamp(2);
    // fused: once the previous item's stores have read the other K/Q buffer
    // and the V buffer, the next item's K/Q tiles and this item's V go there
    // The state pass waits for the first chunk positions: a worker's first
    // item is published here, later ones during the block inverse below.
    const bool publish_now = n_done == 2;
    if (kFused && tid == kPrepIO) {
      io_stamp(0);
      bulk_wait_read_all();
      io_stamp(1);
      if (jn < n_items) issue_kq(nxt, buf ^ 1);
      if (have_prev) issue_v(cur, 0, sm + Lay::V, 8192);
      if (publish_now) publish(prev);
      io_stamp(2);
    }
    __syncthreads();
    if (s_abort) goto teardown;
    if (!mbar_wait(&bar_a, ph)) { flag_status(status, GDN_ERR_TIMEOUT); s_abort = 1; }
    __syncthreads();
    if (s_abort) goto teardown;
    stamp(3);
    tc_fence_after();
    {  // Q^ rows over Q (the Gram MMA has finished reading it)
      const int c = tid;
      uint8_t* qs = kq + (c >> 6) * 16384 + 8192;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(qs + sw_chunk(c & 63, ch)) =
            make_uint4(qv[ch][0], qv[ch][1], qv[ch][2], qv[ch][3]);
    }
    {
      uint32_t g[32];
      tmem_ld32(tmem + lane_off + 32 * hv, g);
      tmem_ld_wait();
      const int row = 32 * quarter + lane;
      if (kSide) {   // the raw Gram rows (K K^T, then Q K^T), zero past the valid rows
        const int r = row & (kC - 1);
        float* dst = (row < kC ? side.KK : side.QK) + ((size_t)(cur.ci * H + cur.h) * kC + r) * kC +
                     32 * hv;
#pragma unroll
        for (int j4 = 0; j4 < 32; j4 += 4) {
          float4 o;
          o.x = (r < L && 32 * hv + j4 < L) ? __uint_as_float(g[j4]) : 0.f;
          o.y = (r < L && 32 * hv + j4 + 1 < L) ? __uint_as_float(g[j4 + 1]) : 0.f;
          o.z = (r < L && 32 * hv + j4 + 2 < L) ? __uint_as_float(g[j4 + 2]) : 0.f;
          o.w = (r < L && 32 * hv + j4 + 3 < L) ? __uint_as_float(g[j4 + 3]) : 0.f;
          *reinterpret_cast<float4*>(dst + j4) = o;
        }
      }
      if (row < kC) {   // A = strict_lower(beta_r Gam_rj k_r.k_j), columns 32hv .. 32hv+31
        const float Gr = sG[row], br = sB[row];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int jc = 32 * hv + jj;
          sA[row * kLd + jc] = jc < row ? br * exp_fast(Gr - sG[jc]) * __uint_as_float(g[jj]) : 0.f;
        }
      } else {          // P^ = lower(Gam_rj q_r.k_j) / sqrt(dk), chunks 4hv .. 4hv+3 of row r
        const int r = row - kC;
        const float Gr = sG[r];
#pragma unroll
        for (int cq = 0; cq < 4; ++cq) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j0 = 32 * hv + 8 * cq + 2 * e, j1 = j0 + 1;
            const float p0 = (j0 <= r && r < L) ? kScale * exp_fast(Gr - sG[j0]) * __uint_as_float(g[8 * cq + 2 * e]) : 0.f;
            const float p1 = (j1 <= r && r < L) ? kScale * exp_fast(Gr - sG[j1]) * __uint_as_float(g[8 * cq + 2 * e + 1]) : 0.f;
            w[e] = pack_bf16(p0, p1);
            if (kSide)
              *reinterpret_cast<float2*>(side.Ph + ((size_t)(cur.ci * H + cur.h) * kC + r) * kC + j0) =
                  make_float2(p0, p1);
          }
          uint8_t* pdst = kFused ? sm + Lay::PS : img + kImgP;
          *reinterpret_cast<uint4*>(pdst + sw_chunk(r, 4 * hv + cq)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    // fused: P^ out; split: Q^ out, then V into the Q slots
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == kPrepIO) {
      io_stamp(3);
      if (kFused) {
        tma_store_1d(img + kImgP, sm + Lay::PS, 8192);
        bulk_commit();
      } else {
        for (int b = 0; b < 4; ++b)
          tma_store_1d(img + kImgWQ + b * 16384 + 8192, kq + b * 16384 + 8192, 8192);
        bulk_commit();
        bulk_wait_read_all();
        issue_v(cur, 0, kq + 8192, 16384);
      }
      io_stamp(4);
    }

    stamp(4);
    // ---- T = (I + A)^{-1}: 16 x 16 diagonal inverses, then two levels of
    //      [[T1, 0], [X, T2]] with X = -T2 A21 T1
    // (forward substitution per column c of block b; four partial sums keep
    // the dependent chain from x[r-1] to x[r] at one FMA and two adds)
    if (tid < 64) {
      const int b = tid >> 4, c = tid & 15, o = 16 * b;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) x[r] = r == c ? 1.f : 0.f;
#pragma unroll
      for (int r = 1; r < 16; ++r) {
        const float* arow = sA + (o + r) * kLd + o;
        float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int jc = 0; jc < r; ++jc) p[jc & 3] = fmaf(arow[jc], x[jc], p[jc & 3]);
        if (r > c) x[r] = -((p[0] + p[1]) + (p[2] + p[3]));
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) sT[(o + r) * kLd + o + c] = x[r];
    } else if (kFused && tid == kPrepIO && have_prev && !publish_now) {
      // meanwhile: every store of the previous item (all groups but this
      // item's P^) has landed, so it can be published
      io_stamp(5);
      bulk_wait_all_but_newest();
      fence_proxy_async_global();
      st_release_gpu(ready + prev.ci * H + prev.h, 1u);
      io_stamp(6);
    }
    __syncthreads();
    {  // level 1, blocks p = 0, 1: Y = A[16(2p+1):, 16(2p):] T_{2p};  T_off = -T_{2p+1} Y
      const int p = tid >> 7, c = tid & 15, r0 = (tid >> 4) & 7;
      const int ro = 16 * (2 * p + 1), co = 16 * (2 * p);
      float y0 = 0.f, y1 = 0.f;
#pragma unroll
      for (int k4 = 0; k4 < 16; k4 += 4) {
        const float4 a0 = *reinterpret_cast<const float4*>(sA + (ro + r0) * kLd + co + k4);
        const float4 a1 = *reinterpret_cast<const float4*>(sA + (ro + r0 + 8) * kLd + co + k4);
        const float t0 = sT[(co + k4) * kLd + co + c], t1 = sT[(co + k4 + 1) * kLd + co + c];
        const float t2 = sT[(co + k4 + 2) * kLd + co + c], t3 = sT[(co + k4 + 3) * kLd + co + c];
        y0 = fmaf(a0.x, t0, fmaf(a0.y, t1, fmaf(a0.z, t2, fmaf(a0.w, t3, y0))));
        y1 = fmaf(a1.x, t0, fmaf(a1.y, t1, fmaf(a1.z, t2, fmaf(a1.w, t3, y1))));
      }
      sY1[p * 256 + r0 * 16 + c] = y0;
      sY1[p * 256 + (r0 + 8) * 16 + c] = y1;
      __syncthreads();
      float z0 = 0.f, z1 = 0.f;
#pragma unroll
      for (int k4 = 0; k4 < 16; k4 += 4) {
        const float4 b0 = *reinterpret_cast<const float4*>(sT + (ro + r0) * kLd + ro + k4);
        const float4 b1 = *reinterpret_cast<const float4*>(sT + (ro + r0 + 8) * kLd + ro + k4);
        const float u0 = sY1[p * 256 + k4 * 16 + c], u1 = sY1[p * 256 + (k4 + 1) * 16 + c];
        const float u2 = sY1[p * 256 + (k4 + 2) * 16 + c], u3 = sY1[p * 256 + (k4 + 3) * 16 + c];
        z0 = fmaf(b0.x, u0, fmaf(b0.y, u1, fmaf(b0.z, u2, fmaf(b0.w, u3, z0))));
        z1 = fmaf(b1.x, u0, fmaf(b1.y, u1, fmaf(b1.z, u2, fmaf(b1.w, u3, z1))));
      }
      sT[(ro + r0) * kLd + co + c] = -z0;
      sT[(ro + r0 + 8) * kLd + co + c] = -z1;
    }
    __syncthreads();
    {  // level 2: Y = A[32:, :32] T[:32, :32];  T[32:, :32] = -T[32:, 32:] Y
      const int c = tid & 31, r0 = tid >> 5;
      float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
      for (int k4 = 0; k4 < 32; k4 += 4) {
        const float t0 = sT[k4 * kLd + c], t1 = sT[(k4 + 1) * kLd + c];
        const float t2 = sT[(k4 + 2) * kLd + c], t3 = sT[(k4 + 3) * kLd + c];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 a = *reinterpret_cast<const float4*>(sA + (32 + r0 + 8 * m) * kLd + k4);
          y[m] = fmaf(a.x, t0, fmaf(a.y, t1, fmaf(a.z, t2, fmaf(a.w, t3, y[m]))));
        }
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) sY2[(r0 + 8 * m) * 33 + c] = y[m];
      __syncthreads();
      float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
      for (int k4 = 0; k4 < 32; k4 += 4) {
        const float u0 = sY2[k4 * 33 + c], u1 = sY2[(k4 + 1) * 33 + c];
        const float u2 = sY2[(k4 + 2) * 33 + c], u3 = sY2[(k4 + 3) * 33 + c];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 b = *reinterpret_cast<const float4*>(sT + (32 + r0 + 8 * m) * kLd + 32 + k4);
          z[m] = fmaf(b.x, u0, fmaf(b.y, u1, fmaf(b.z, u2, fmaf(b.w, u3, z[m]))));
        }
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) sT[(32 + r0 + 8 * m) * kLd + c] = -z[m];
    }
    __syncthreads();
    stamp(5);
    // T_w = T diag(beta gamma), T_u = T diag(beta): K-major bf16 images over the dead A tile
    {
      const int r = tid >> 2, c2 = tid & 3;
#pragma unroll
      for (int cq = 0; cq < 2; ++cq) {
        const int ch = 2 * c2 + cq;
        uint32_t ww[4], uu[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j0 = ch * 8 + 2 * e, j1 = j0 + 1;
          const float t0v = j0 <= r ? sT[r * kLd + j0] : 0.f;
          const float t1v = j1 <= r ? sT[r * kLd + j1] : 0.f;
          const float b0 = sB[j0], b1 = sB[j1];
          ww[e] = pack_bf16(t0v * b0 * sGam[j0], t1v * b1 * sGam[j1]);
          uu[e] = pack_bf16(t0v * b0, t1v * b1);
          if (kSide) {   // T, T diag(beta gamma), T diag(beta) in fp32
            const size_t o = ((size_t)(cur.ci * H + cur.h) * kC + r) * kC + j0;
            *reinterpret_cast<float2*>(side.Tm + o) = make_float2(t0v, t1v);
            *reinterpret_cast<float2*>(side.TmB + o) =
                make_float2(t0v * b0 * sGam[j0], t1v * b1 * sGam[j1]);
            *reinterpret_cast<float2*>(side.TmU + o) = make_float2(t0v * b0, t1v * b1);
          }
        }
        *reinterpret_cast<uint4*>(sm + Lay::TW + sw_chunk(r, ch)) = make_uint4(ww[0], ww[1], ww[2], ww[3]);
        *reinterpret_cast<uint4*>(sm + Lay::TU + sw_chunk(r, ch)) = make_uint4(uu[0], uu[1], uu[2], uu[3]);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    stamp(6);
    // ---- W^T = K^T T_w^T and U~^T = V^T T_u^T: two 128-row halves of W^T
    //      and of each 256-column block vh of V (dv = 512: a second pass
    //      over the second block, once the first block's U~^T has left)
    for (int vh = 0; vh * kDK < dv; ++vh) {
      if (vh > 0 && tid == kPrepIO) {
        bulk_wait_read_all();
        issue_v(cur, vh, kFused ? sm + Lay::V : kq + 8192, kFused ? 8192 : 16384);
      }
      if (conv) {   // v: convolution + SiLU in place
        conv_tile(cur, kFused ? sm + Lay::V : kq + 8192, kFused ? 8192 : 16384,
                  (int64_t)(2 * H + cur.h) * kDK + kDK * vh, false, false, &bar_v, vph);
        fence_proxy_async_smem();
        __syncthreads();
      }
      if (tid == 0) {
        if (!mbar_wait(&bar_v, vph)) {
          s_abort = 1;
        } else {
          tc_fence_after();
          const uint32_t idesc = idesc_bf16(128, 64, 1, 0);
          const uint32_t kqa = smem_u32(kq);
          // V's 64-column blocks: own buffer (fused) or the Q slots (split)
          const uint32_t va = kFused ? smem_u32(sm + Lay::V) : kqa + 8192;
          const uint32_t vblk = kFused ? 8192 : 16384;
          const uint32_t tw = smem_u32(sm + Lay::TW), tu = smem_u32(sm + Lay::TU);
          for (int hh = 0; hh < 2; ++hh) {
            if (vh == 0)
              for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + hh * 64, smem_desc(kqa + hh * 32768 + s * 2048, 16384, 1024, kSwizzle128B),
                         smem_desc(tw + s * 32, 16, 1024, kSwizzle128B), idesc, s > 0);
            for (int s = 0; s < 4; ++s)
              mma_bf16(tmem + 128 + hh * 64,
                       smem_desc(va + hh * 2 * vblk + s * 2048, vblk, 1024, kSwizzle128B),
                       smem_desc(tu + s * 32, 16, 1024, kSwizzle128B), idesc, s > 0);
          }
          mma_commit(&bar_bc);
        }
      }
      vph ^= 1u;
      __syncthreads();
      if (s_abort) goto teardown;
      if (!mbar_wait(&bar_bc, bcph)) { flag_status(status, GDN_ERR_TIMEOUT); s_abort = 1; }
      bcph ^= 1u;
      __syncthreads();
      if (s_abort) goto teardown;
      if (vh == 0) stamp(7);
      tc_fence_after();
      // W rows c over the K slots (K consumed); U~^T rows over V (consumed):
      // fused, the V buffer in image layout, split, the Q slots
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t c = 128 * hh + 32 * quarter + lane;   // d_k row of W^T / d_v row of U~^T
#pragma unroll
        for (int part = 0; part < 2; ++part) {               // 0: W, 1: U~^T
          if (part == 0 && vh > 0) continue;
          uint32_t g[32];
          tmem_ld32(tmem + lane_off + part * 128 + hh * 64 + 32 * hv, g);
          tmem_ld_wait();
          uint8_t* base;    // 128-byte rows from here, swizzled by row
          uint32_t row;
          if (part == 0) {
            base = kq + (c >> 6) * 16384;
            row = c & 63;
          } else if (kFused) {
            base = sm + Lay::V + hh * kImgHalf;
            row = c & 127;
          } else {
            base = kq + (c >> 6) * 16384 + 8192;
            row = c & 63;
          }
#pragma unroll
          for (int cq = 0; cq < 4; ++cq) {
            const uint32_t w0 = pack_bf16(__uint_as_float(g[8 * cq]), __uint_as_float(g[8 * cq + 1]));
            const uint32_t w1 = pack_bf16(__uint_as_float(g[8 * cq + 2]), __uint_as_float(g[8 * cq + 3]));
            const uint32_t w2 = pack_bf16(__uint_as_float(g[8 * cq + 4]), __uint_as_float(g[8 * cq + 5]));
            const uint32_t w3 = pack_bf16(__uint_as_float(g[8 * cq + 6]), __uint_as_float(g[8 * cq + 7]));
            *reinterpret_cast<uint4*>(base + sw_chunk(row, 4 * hv + cq)) = make_uint4(w0, w1, w2, w3);
          }
        }
      }
      if (tid < kC) {
        const float d = tid < L ? exp_fast(sG[L - 1] - sG[tid]) : 0.f;
        if (kFused) {
          for (int hh = 0; hh < 2; ++hh) {
            float* blk = reinterpret_cast<float*>(sm + Lay::V + hh * kImgHalf + kImgDecay);
            blk[tid] = d;
            blk[64 + tid] = sG[tid];
          }
        } else if (vh == 0) {
          sDecay[tid] = d;
          sDecay[64 + tid] = sG[tid];
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == kPrepIO) {
        // U~^T slices 2 vh and 2 vh + 1 of the image
        uint8_t* uimg = img + kImgU0 + 2 * vh * kImgHalf;
        if (kFused) {
          if (vh == 0) tma_store_1d(img + kImgWQ, kq, 65536);
          tma_store_1d(uimg, sm + Lay::V, (uint32_t)(2 * kImgHalf));
        } else {
          for (int b = 0; b < 4; ++b) {
            if (vh == 0) tma_store_1d(img + kImgWQ + b * 16384, kq + b * 16384, 8192);
            tma_store_1d(uimg + (b >> 1) * kImgHalf + (b & 1) * 8192, kq + b * 16384 + 8192, 8192);
          }
          for (int hh = 0; hh < 2; ++hh) tma_store_1d(uimg + hh * kImgHalf + kImgDecay, sDecay, 512);
        }
        bulk_commit();
        io_stamp(7);
      }
    }
    stamp(8);
    prev = cur;
    have_prev = true;
    cur = nxt;
    j = jn;
    a_cur = a_nx;
    b_cur = b_nx;
    if (kFused) buf ^= 1;
    ph ^= 1u;
  }

teardown:
  if (tid == kPrepIO) {
    if (kFused && have_prev && !s_abort) publish(prev);
    bulk_wait_all();   // the stores read shared memory: finish before the CTA exits
    if (s_abort) {     // let copies still in flight land
      flag_status(status, GDN_ERR_TIMEOUT);
      for (int b = 0; b < kBufs; ++b)
        if (n_kq[b]) mbar_wait(&bar_kq[b], (n_kq[b] - 1) & 1, 100000000ull);
      if (n_v) mbar_wait(&bar_v, (n_v - 1) & 1, 100000000ull);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
  if (timed) timeline[kWorkerTimes + 2 * worker + 1] = globaltimer_ns();
}

// =========================================================== state pass
constexpr int kStateThreads = 256;
constexpr uint32_t kS_WQ = 0;         // 2 x 64 KB: [W (32 KB) | Q^ (32 KB)] per buffer
constexpr uint32_t kS_KP = 131072;    // 2 x 40 KB: [K (32 KB, MN-major) | P^ (8 KB)] per buffer
constexpr uint32_t kS_UT = 212992;    // 16.5 KB: U~^T rows of this half + decay block
constexpr uint32_t kS_END = 229888;
constexpr uint32_t kStateSmem = kS_END + 1024;
// TMEM columns: D_U (fp32), D_O (fp32), the bf16 A-operand copy of S (2 per
// column), D_S (fp32).  After the U epilogue the D_U columns hold bf16 A
// operands: each half [32h, 32h+32) of D_U is overwritten only by the warps
// that read it, with U for rows r in [32h, 32h+32) in its first 16 columns
// and d*U for the same rows in its last 16.
constexpr uint32_t kT_U = 0, kT_O = 64, kT_SA = 128, kT_S = 256;
__device__ __forceinline__ uint32_t col_U(int s) { return 32u * (s >> 1) + 8u * (s & 1); }
__device__ __forceinline__ uint32_t col_dU(int s) { return col_U(s) + 16u; }

// One state unit: sequence n, head h, rows [128 half, 128 half + 128) of S.
// kFused: the images of each chunk are acquired through its ready flag.
template <bool kFused>
__device__ __forceinline__ void state_role(uint8_t* sm, const CUtensorMap* tm_k,
                                           const float* __restrict__ S0,
                                           __nv_bfloat16* __restrict__ out,
                                           float* __restrict__ S_final, const SeqMap& map,
                                           int32_t H, const uint8_t* __restrict__ scratch,
                                           const uint32_t* ready, unsigned* status,
                                           uint64_t* __restrict__ trace, int32_t trace_chunks,
                                           int32_t dv, int n, int h, int slice,
                                           float* __restrict__ sdump, const NormGate& ng,
                                           bool a_chain = false) {
  const int unit = (n * H + h) * (dv / 128) + slice;
  const bool timed = trace && threadIdx.x == 0 && unit < kMaxTracedUnits;
  if (timed) trace[kUnitTimes + 3 * unit] = globaltimer_ns();
  const float* sD = reinterpret_cast<const float*>(sm + kS_UT + kImgDecay);   // d_r, then G_r
  __shared__ uint64_t bar_wq[2], bar_kp[2], bar_p[2], bar_u, bar_m1, bar_m1b, bar_m2, bar_mo;
  // (fused) chunks [cb, s_ready_hi) of this unit are known to be published;
  // written only by warp 1 at the top of a chunk, read by the loaders after
  // the chunk's first barrier
  __shared__ long long s_ready_hi;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  const bool norm = ng.gate != nullptr;   // the read-out with the gated RMSNorm

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, colhalf = warp >> 2;
  const uint32_t iloc = 32 * quarter + lane;            // TMEM lane = local row of S
  const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
  const int64_t cb = map.chunk_begin(n), ce = map.chunk_end(n);
  const int64_t s_begin = map.seq_begin(n), s_end = map.seq_end(n);
  // optional phase timeline (test hook): thread 0 of unit (0, 0, 0) stamps
  // its SM cycle counter at 12 points of each of its first trace_chunks chunks
  const bool tracing = trace && tid == 0 && n == 0 && h == 0 && slice == 0;
  auto stamp = [&](int64_t it, int k) {
    if (tracing && it < trace_chunks) trace[it * 12 + k] = clock64();
  };

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_wq[b], 1);
      mbar_init(&bar_kp[b], 1);
      mbar_init(&bar_p[b], 1);
    }
    mbar_init(&bar_u, 1);
    mbar_init(&bar_m1, 1);
    mbar_init(&bar_m1b, 1);
    mbar_init(&bar_m2, 1);
    mbar_init(&bar_mo, 1);
    fence_barrier_init();
    s_abort = 0;
    s_ready_hi = cb;
    prefetch_tensormap(tm_k);
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);

  // master state: this thread's 128 columns of row iloc (fp32, registers)
  float S[128];
  // S0 / S_final point at this unit's [H][dv][dk] block
  const size_t srow = (((size_t)h) * dv + 128 * slice + iloc) * kDK + 128 * colhalf;
  if (S0) {
    const float4* p = reinterpret_cast<const float4*>(S0 + srow);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float4 t = p[j];
      S[4 * j] = t.x; S[4 * j + 1] = t.y; S[4 * j + 2] = t.z; S[4 * j + 3] = t.w;
    }
  } else {
    // zero, or the identity (an A chain: the product of the chunks'
    // transitions, rows 0 .. dk-1)
    const uint32_t row = 128 * slice + iloc, col0 = 128 * colhalf;
#pragma unroll
    for (int j = 0; j < 128; ++j) S[j] = a_chain && row == col0 + j ? 1.f : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  // bf16 copy of S into TMEM: one packed column holds two state columns
  auto store_S_operand = [&]() {
#pragma unroll
    for (int hq = 0; hq < 2; ++hq) {
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = pack_bf16(S[64 * hq + 2 * j], S[64 * hq + 2 * j + 1]);
      tmem_st32(tmem + lane_off + kT_SA + 64 * colhalf + 32 * hq, r);
    }
    tmem_st_wait();
  };
  store_S_operand();

  // A unit whose outputs nobody reads (the long-sequence form's B and A
  // chains) needs neither Q^ nor P^: its MMA-1 is N = 64 over W alone, it
  // skips MMA-O and the output epilogue, and an A chain also skips U~ (it
  // reads only the decay block), so its chunk loads 80.5 KB (64.5 KB)
  // instead of 120.5 KB.
  const bool nout = out == nullptr;
  auto img_of = [&](int64_t ci) { return scratch + (size_t)(ci * H + h) * img_stride(dv); };
  auto t0_of = [&](int64_t ci) { return (int32_t)(s_begin + (ci - cb) * kC); };
  auto flag_of = [&](int64_t ci) { return ready + ci * H + h; };
  auto issue_wq = [&](int64_t ci, int buf) {   // W and Q^ are adjacent in the image
    if (nout) {   // the four 8 KB blocks of W, each followed by Q^'s in the image
      mbar_arrive_expect_tx(&bar_wq[buf], 32768);
      for (int b = 0; b < 4; ++b)
        tma_load_1d(sm + kS_WQ + buf * 65536 + b * 16384, img_of(ci) + kImgWQ + b * 16384, 8192,
                    &bar_wq[buf]);
      return;
    }
    mbar_arrive_expect_tx(&bar_wq[buf], 65536);
    tma_load_1d(sm + kS_WQ + buf * 65536, img_of(ci) + kImgWQ, 65536, &bar_wq[buf]);
  };
  auto issue_k = [&](int64_t ci, int buf) {   // K tile of the chunk, straight from the input
    mbar_arrive_expect_tx(&bar_kp[buf], 32768);
    tma_load_4d(sm + kS_KP + buf * 40960, tm_k, 0, t0_of(ci), 0, h, &bar_kp[buf]);
  };
  auto issue_p = [&](int64_t ci, int buf) {
    mbar_arrive_expect_tx(&bar_p[buf], 8192);
    tma_load_1d(sm + kS_KP + buf * 40960 + 32768, img_of(ci) + kImgP, 8192, &bar_p[buf]);
  };
  auto issue_u = [&](int64_t ci) {    // this half's U~^T rows and the decay block
    if (a_chain) {                    // the decay block alone
      mbar_arrive_expect_tx(&bar_u, (uint32_t)(kImgHalf - kImgDecay));
      tma_load_1d(sm + kS_UT + kImgDecay, img_of(ci) + kImgU0 + slice * kImgHalf + kImgDecay,
                  (uint32_t)(kImgHalf - kImgDecay), &bar_u);
      return;
    }
    mbar_arrive_expect_tx(&bar_u, (uint32_t)kImgHalf);
    tma_load_1d(sm + kS_UT, img_of(ci) + kImgU0 + slice * kImgHalf, (uint32_t)kImgHalf, &bar_u);
  };
  auto warm_l2 = [&](int64_t ci) {    // the whole image of a later chunk (split form)
    prefetch_l2(img_of(ci), (uint32_t)img_stride(dv));
  };
  // Loads are issued by single threads of warps 1, 2 and 3 (thread 0 issues
  // the MMAs), so that each one's issue work fits in the time MMA-2 takes.
  // Each counts the phases it started on its load barriers, for a clean exit
  // after a timeout.
  constexpr int kLoaderA = 32;   // K, one chunk ahead; polls the ready flags
  constexpr int kLoaderB = 64;   // W / Q^, two chunks ahead, and the L2 warm-up
  constexpr int kLoaderC = 96;   // P^, U~^T and the decay block, one chunk ahead
  uint32_t n_wq[2] = {0, 0}, n_kp[2] = {0, 0}, n_p[2] = {0, 0}, n_u = 0;
  int64_t wq_next = cb;          // (kLoaderB) first chunk whose W / Q^ is not issued yet
  // Ready flags (fused form).  A poll reads the flags of eight chunks from
  // `from` with relaxed loads (one round trip) and, when the first few are
  // set, makes what they published visible with one acquire fence; it
  // returns the new bound of known-published chunks.  Warp 1 polls 32 chunks
  // at a time at the top of a chunk, while MMA-1 runs and warps 1-3 have
  // nothing else to do, and shares the bound; the loaders' own checks then
  // cost nothing unless the per-chunk work has fallen behind.
  auto poll_from = [&](int64_t from) -> int64_t {
    uint32_t v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = from + k < ce ? ld_relaxed_gpu(flag_of(from + k)) : 0u;
    int k = 0;
    bool run = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      run = run && v[i] != 0;
      k += run;
    }
    if (k > 0) {
      fence_acq_rel_gpu();
      fence_proxy_async_global();
    }
    return from + k;
  };
  int64_t my_hi = cb;   // this thread's own bound
  auto is_ready = [&](int64_t ci, bool wait) -> bool {
    if (!kFused || ci < my_hi) return true;
    const int64_t sh = (int64_t)*reinterpret_cast<volatile long long*>(&s_ready_hi);
    if (ci < sh) {   // published as seen by the first loader before the last barrier
      my_hi = sh;
      fence_proxy_async_global();
      return true;
    }
    my_hi = poll_from(my_hi > sh ? my_hi : sh);
    if (ci < my_hi || !wait) return ci < my_hi;
    const uint64_t t_start = globaltimer_ns();
    do {
      __nanosleep(64);
      my_hi = poll_from(my_hi);
      if (ci < my_hi) return true;
    } while (globaltimer_ns() - t_start < kReadyWaitNs);
    return false;
  };
  auto load_k = [&](int64_t ci, int buf) -> bool {   // (kLoaderA)
    if (!is_ready(ci, true)) return false;
    issue_k(ci, buf); ++n_kp[buf];
    return true;
  };
  auto load_pu = [&](int64_t ci, int buf) -> bool {   // (kLoaderC)
    if (!is_ready(ci, true)) return false;
    if (!nout) {
      issue_p(ci, buf); ++n_p[buf];
    }
    issue_u(ci); ++n_u;
    return true;
  };
  // (kLoaderB) W / Q^ of every chunk up to `must` (waiting for its flag) and
  // of the chunk after it if that is already published; the buffer of chunk
  // c is free once MMA-1 of chunk c - 2 has finished (m1_done).
  auto load_wq = [&](int64_t must, bool m1_done) -> bool {
    while (wq_next < ce && wq_next <= must + 1) {
      if (wq_next == must + 1) {
        if (!m1_done || !is_ready(wq_next, false)) break;
      } else if (!is_ready(wq_next, true)) {
        return false;
      }
      const int b = (int)((wq_next - cb) & 1);
      issue_wq(wq_next, b); ++n_wq[b];
      ++wq_next;
    }
    return true;
  };
  if (cb < ce && ((tid == kLoaderA && !load_k(cb, 0)) || (tid == kLoaderC && !load_pu(cb, 0)))) {
    flag_status(status, GDN_ERR_TIMEOUT);
    s_abort = 1;
  }
  if (tid == kLoaderB && cb < ce) {
    if (!load_wq(cb, true)) {
      flag_status(status, GDN_ERR_TIMEOUT);
      s_abort = 1;
    }
    if (!kFused && cb + 1 < ce) warm_l2(cb + 1);
    if (!kFused && cb + 2 < ce) warm_l2(cb + 2);
  }
  tc_fence_before();
  __syncthreads();
  int prev_L = 0;
  int64_t prev_t0 = 0;
  // rows of out for the previous chunk, staged in its (consumed) K / P^ buffer
  // as [r][128] bf16 (256 B per row, this unit's half of the row of out);
  // consecutive threads of warps 4-7 move consecutive 16-byte pieces, so each
  // warp store covers two whole 256-byte row segments.  (Warp 0 is issuing
  // MMA-1 then; warps 1-3 hold the loader threads, whose acquire fences
  // would otherwise wait for these stores to drain.)
  //
  // (norm) The 16 threads of a row also sum the squares of its 128 bf16
  // values (the values a separate pass would read) and one of them stores the
  // row's partial sum; Eq. 20 itself runs after the chain (norm_tail).
  auto copy_out_prev = [&](int prev_buf) {
    if (!out) return;   // a unit whose outputs nobody reads
    const uint8_t* stage = sm + kS_KP + prev_buf * 40960;
    for (int p = tid - 128; p < 16 * prev_L; p += kStateThreads - 128) {
      if (p < 0) break;
      const int r = p >> 4, c16 = p & 15;
      const uint4 v = *reinterpret_cast<const uint4*>(stage + r * 256 + c16 * 16);
      *reinterpret_cast<uint4*>(out + ((prev_t0 + r) * H + h) * dv + 128 * slice + 8 * c16) = v;
      if (norm && !(kFused && ng.flags)) {   // whole 16-lane halves of a warp share a row
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        float ssum = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = bf16_lo(w4[e]), b = bf16_hi(w4[e]);
          ssum = fmaf(a, a, ssum);
          ssum = fmaf(b, b, ssum);
        }
        const unsigned half = 0xffffu << (lane & 16);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) ssum += __shfl_xor_sync(half, ssum, o);
        if (c16 == 0) ng.part[((prev_t0 + r) * H + h) * 2 + slice] = ssum;
      }
    }
  };

  for (int64_t ci = cb; ci < ce && !s_abort; ++ci) {
    const int64_t it = ci - cb;
    const uint32_t par = (uint32_t)(it & 1);
    const int buf = (int)(it & 1);
    const uint32_t bpar = (uint32_t)((it >> 1) & 1);
    const int64_t t0 = s_begin + it * kC;
    const int L = (int)min((int64_t)kC, s_end - t0);

    // 1. [D_U | D_O] = S [W | Q^]^T (commit m1 and m1b); A = S from TMEM
    stamp(it, 0);
    // (fused) warp 1 refreshes the shared bound when fewer than eight chunks
    // ahead are known: one flag per lane, the run of published chunks from
    // the bound by ballot, one acquire fence for all of them
    if (kFused && warp == 1) {
      const int64_t hi = *reinterpret_cast<volatile long long*>(&s_ready_hi);
      if (hi < (ci + 8 < ce ? ci + 8 : ce)) {
        const uint32_t f = hi + lane < ce ? ld_relaxed_gpu(flag_of(hi + lane)) : 0u;
        const unsigned set = __ballot_sync(0xffffffffu, f != 0);
        const int k = set == 0xffffffffu ? 32 : __ffs(~set) - 1;
        if (k > 0) {
          fence_acq_rel_gpu();
          fence_proxy_async_global();
        }
        __syncwarp();
        if (lane == 0) s_ready_hi = hi + k;
      }
    }
    if (timed && it == 0) trace[kUnitTimes + 3 * unit + 1] = globaltimer_ns();
    if (tid == 0) {
      if (!mbar_wait(&bar_wq[buf], bpar)) {
        s_abort = 1;
      } else {
        tc_fence_after();
        // [D_U | D_O] = S [W | Q^]^T : one N = 128 operand (MN-major; for the
        // 16 K-rows of step s, block s / 4 of W at 16 KB strides and the
        // matching Q^ block 8 KB after it)
        const uint32_t id1 = idesc_bf16(128, nout ? 64 : 128, 0, 1);
        const uint32_t sW = smem_u32(sm + kS_WQ + buf * 65536);
        for (int s = 0; s < 16; ++s)
          mma_bf16_ts(tmem + kT_U, tmem + kT_SA + 8 * s,
                      smem_desc(sW + (s >> 2) * 16384 + (s & 3) * 2048, 8192, 1024, kSwizzle128B),
                      id1, s > 0);
        mma_commit(&bar_m1);
        mma_commit(&bar_m1b);
      }
    }
    stamp(it, 1);
    // the previous chunk's output rows go out while MMA-1 runs
    if (it > 0) copy_out_prev(buf ^ 1);
    // (optional) this chunk's start state, for the backward's forward re-run
    if (sdump) {
      const size_t v = 128 * slice + iloc;
      if (tiled_states(dv)) {   // bf16 tiles; lanes: consecutive rows, 256 contiguous bytes a store
        uint2* p = reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(sdump) +
                                            (size_t)(ci * H + h) * dv * kDK) +
                   (size_t)32 * colhalf * dv + v;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          p[(size_t)j * dv] = make_uint2(pack_bf16(S[4 * j], S[4 * j + 1]),
                                         pack_bf16(S[4 * j + 2], S[4 * j + 3]));
      } else {
        float* base = sdump + (size_t)(ci * H + h) * dv * kDK;
        float4* p = reinterpret_cast<float4*>(base + v * kDK + 128 * colhalf);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          p[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
      }
    }
    // 2. U = U~ - D_U (columns r = 32 colhalf ..), and d_r U: bf16 A operands in TMEM
    float gC = 0.f;
    if (!mbar_wait(&bar_m1, par) || !mbar_wait(&bar_u, par)) {
      flag_status(status, GDN_ERR_TIMEOUT);
      s_abort = 1;
    } else {
      tc_fence_after();
      uint32_t g[32];
      tmem_ld32(tmem + lane_off + kT_U + 32 * colhalf, g);
      tmem_ld_wait();
      stamp(it, 8);
      gC = exp_fast(sD[64 + L - 1]);
      uint32_t ua[16], ud[16];
#pragma unroll
      for (int cq = 0; cq < 4; ++cq) {
        const uint4 ut = *reinterpret_cast<const uint4*>(sm + kS_UT + sw_chunk(iloc, 4 * colhalf + cq));
        const uint32_t uw[4] = {ut.x, ut.y, ut.z, ut.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 8 * cq + 2 * e, r = 32 * colhalf + j;
          // an A chain drops U~ (the homogeneous part of the recurrence)
          const float u0 = (a_chain ? 0.f : bf16_lo(uw[e])) - __uint_as_float(g[j]);
          const float u1 = (a_chain ? 0.f : bf16_hi(uw[e])) - __uint_as_float(g[j + 1]);
          const float d0 = sD[r], d1 = sD[r + 1];
          ua[4 * cq + e] = pack_bf16(u0, u1);
          ud[4 * cq + e] = pack_bf16(u0 * d0, u1 * d1);
        }
      }
      tmem_st16(tmem + lane_off + kT_U + 32 * colhalf, ua);
      tmem_st16(tmem + lane_off + kT_U + 32 * colhalf + 16, ud);
      tmem_st_wait();
    }
    stamp(it, 2);
    tc_fence_before();
    __syncthreads();
    if (s_abort) break;
    stamp(it, 3);
    // (fused read-out) every kReadoutStep chunks: the rows of chunks
    // [cb, ci) are out (copied before the barrier).  A release waits for the
    // CTA's stores to drain, so it is not made every chunk.
    if (kFused && ng.flags && it > 0 && it % kReadoutStep == 0 && tid == 128)
      st_release_gpu(ng.flags + unit, (uint32_t)it);

    // 3. D_S = (dU)^T K (commit m2) ; D_O += U^T P^^T (commit mo)
    if (tid == 0) {
      if (!mbar_wait(&bar_kp[buf], bpar) || (!nout && !mbar_wait(&bar_p[buf], bpar))) {
        s_abort = 1;
      } else {
        tc_fence_after();
        const uint32_t id2 = idesc_bf16(128, 256, 0, 1), idO = idesc_bf16(128, 64, 0, 0);
        const uint32_t sK = smem_u32(sm + kS_KP + buf * 40960), sP = sK + 32768;
        for (int s = 0; s < 4; ++s)
          mma_bf16_ts(tmem + kT_S, tmem + kT_U + col_dU(s),
                      smem_desc(sK + s * 2048, 8192, 1024, kSwizzle128B), id2, s > 0);
        mma_commit(&bar_m2);
        if (!nout) {
          for (int s = 0; s < 4; ++s)
            mma_bf16_ts(tmem + kT_O, tmem + kT_U + col_U(s),
                        smem_desc(sP + s * 32, 16, 1024, kSwizzle128B), idO, 1);
          mma_commit(&bar_mo);
        }
      }
    }
    // ... meanwhile the loaders fetch ahead: K / P^ and U~^T of the next
    // chunk (the previous chunk's staging was copied out above and E1 is done
    // with the U~^T buffer), W / Q^ of the next chunk if not yet in flight
    // and of the chunk after it once MMA-1 finished reading this buffer, and
    // (split form) L2 warm-up of a later chunk's image
    if (ci + 1 < ce && ((tid == kLoaderA && !load_k(ci + 1, buf ^ 1)) ||
                        (tid == kLoaderC && !load_pu(ci + 1, buf ^ 1)))) {
      flag_status(status, GDN_ERR_TIMEOUT);
      s_abort = 1;
    }
    if (tid == kLoaderB) {
      if (!kFused && ci + 3 < ce) warm_l2(ci + 3);
      if (ci + 1 < ce) {
        const bool m1_done = ci + 2 < ce ? mbar_wait(&bar_m1b, par) : true;
        if (!m1_done) s_abort = 1;
        if (!load_wq(ci + 1, m1_done)) {
          flag_status(status, GDN_ERR_TIMEOUT);
          s_abort = 1;
        }
      }
    }

    // 4. S = gamma_L S + D_S (fp32) -> bf16 operand copy in TMEM; O -> out
    stamp(it, 4);
    if (!mbar_wait(&bar_m2, par)) {
      flag_status(status, GDN_ERR_TIMEOUT);
      s_abort = 1;
    } else {
      stamp(it, 5);
      tc_fence_after();
      // MMA-1 has finished reading the bf16 state operand (it precedes
      // MMA-2), so each folded group can replace its columns right away.
      // Groups of 16 columns; the load of group q + 1 is in flight while
      // group q is folded.
      if (!mbar_wait(&bar_m1b, par)) s_abort = 1;
      const uint32_t tS = tmem + lane_off + kT_S + 128 * colhalf;
      const uint32_t tA = tmem + lane_off + kT_SA + 64 * colhalf;
      uint32_t g[2][16];
      tmem_ld16(tS, g[0]);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        tmem_ld_wait_regs(g[q & 1]);
        if (q + 1 < 8) tmem_ld16(tS + 16 * (q + 1), g[(q + 1) & 1]);
        uint32_t pk[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float s0 = fmaf(gC, S[16 * q + j], __uint_as_float(g[q & 1][j]));
          const float s1 = fmaf(gC, S[16 * q + j + 1], __uint_as_float(g[q & 1][j + 1]));
          S[16 * q + j] = s0;
          S[16 * q + j + 1] = s1;
          pk[j >> 1] = pack_bf16(s0, s1);
        }
        tmem_st8(tA + 8 * q, pk);
      }
      tmem_st_wait();
      stamp(it, 9);
      if (nout) {
      } else if (!mbar_wait(&bar_mo, par)) {
        flag_status(status, GDN_ERR_TIMEOUT);
        s_abort = 1;
      } else {
        stamp(it, 10);
        tc_fence_after();
        uint32_t g[32];
        tmem_ld32(tmem + lane_off + kT_O + 32 * colhalf, g);
        tmem_ld_wait();
        stamp(it, 11);
        // O^T (row iloc, columns r) -> staging [r][128] bf16 in this chunk's
        // K / P^ buffer, which MMA-2 and MMA-O no longer read
        __nv_bfloat16* so = reinterpret_cast<__nv_bfloat16*>(sm + kS_KP + buf * 40960);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(g[j]), __uint_as_float(g[j + 1]));
          so[(32 * colhalf + j) * 128 + iloc] = pr.x;
          so[(32 * colhalf + j + 1) * 128 + iloc] = pr.y;
        }
      }
    }
    stamp(it, 6);
    tc_fence_before();
    __syncthreads();
    if (s_abort) break;
    stamp(it, 7);

    prev_L = L;
    prev_t0 = t0;
  }
  // the last chunk's output rows
  if (!s_abort && ce > cb) copy_out_prev((int)((ce - cb - 1) & 1));
  if (kFused && ng.flags && ce > cb) {   // and finally all of them
    __syncthreads();
    if (!s_abort && tid == 128) st_release_gpu(ng.flags + unit, (uint32_t)(ce - cb));
  }

  if (!s_abort && S_final) {
    float4* p = reinterpret_cast<float4*>(S_final + srow);
#pragma unroll
    for (int j = 0; j < 32; ++j) p[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
  }
  if ((tid == kLoaderA || tid == kLoaderB || tid == kLoaderC) && s_abort) {   // let copies in flight land
    flag_status(status, GDN_ERR_TIMEOUT);
    const uint64_t lim = 100000000ull;
    for (int b = 0; b < 2; ++b) {
      if (n_wq[b]) mbar_wait(&bar_wq[b], (n_wq[b] - 1) & 1, lim);
      if (n_kp[b]) mbar_wait(&bar_kp[b], (n_kp[b] - 1) & 1, lim);
      if (n_p[b]) mbar_wait(&bar_p[b], (n_p[b] - 1) & 1, lim);
    }
    if (n_u) mbar_wait(&bar_u, (n_u - 1) & 1, lim);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
  // (norm) Eq. 20 over this unit's rows, once both units of the head (the
  // cluster) have stored their outputs and partial sums: an HBM stream of
  // out, gate and out again, off the chain's critical path (units of other
  // sequences are still walking their chains meanwhile).  Every thread takes
  // 16-byte pieces of one column group (tid & 15), kTailRows rows at a time,
  // with all loads of those rows in flight before any is used (the chain's
  // registers are free by now).
  constexpr int kTailRows = 8;
  if (norm && !(kFused && ng.flags)) {
    cluster_sync_all();
    if (out && !s_abort) {
      const int c16 = tid & 15;
      const int col = 128 * slice + 8 * c16;
      float w8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w8[i] = __ldg(ng.w + col + i);
      const float inv_dv = 1.f / (float)dv;
      for (int64_t t = s_begin + (tid >> 4); t < s_end; t += kTailRows * (kStateThreads / 16)) {
        uint4 ov[kTailRows], gv[kTailRows];
        float ps[kTailRows];
#pragma unroll
        for (int u = 0; u < kTailRows; ++u) {
          const int64_t tu = t + u * (kStateThreads / 16);
          if (tu < s_end) {
            const size_t off = ((size_t)tu * H + h) * dv + col;
            ov[u] = *reinterpret_cast<const uint4*>(out + off);
            gv[u] = __ldg(reinterpret_cast<const uint4*>(ng.gate + off));
            const float2 pp = *reinterpret_cast<const float2*>(ng.part + ((size_t)tu * H + h) * 2);
            ps[u] = pp.x + pp.y;
          }
        }
#pragma unroll
        for (int u = 0; u < kTailRows; ++u) {
          const int64_t tu = t + u * (kStateThreads / 16);
          if (tu < s_end) {
            const float rs = rsqrtf(ps[u] * inv_dv + ng.eps);
            const uint32_t o4[4] = {ov[u].x, ov[u].y, ov[u].z, ov[u].w};
            const uint32_t g4[4] = {gv[u].x, gv[u].y, gv[u].z, gv[u].w};
            uint32_t yo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float g0 = bf16_lo(g4[e]), g1 = bf16_hi(g4[e]);
              const float a0 = ng.act == GDN_GATE_SIGMOID ? __fdividef(1.f, 1.f + __expf(-g0))
                                                          : __fdividef(g0, 1.f + __expf(-g0));
              const float a1 = ng.act == GDN_GATE_SIGMOID ? __fdividef(1.f, 1.f + __expf(-g1))
                                                          : __fdividef(g1, 1.f + __expf(-g1));
              yo[e] = pack_bf16(bf16_lo(o4[e]) * rs * w8[2 * e] * a0,
                                bf16_hi(o4[e]) * rs * w8[2 * e + 1] * a1);
            }
            *reinterpret_cast<uint4*>(out + ((size_t)tu * H + h) * dv + col) =
                make_uint4(yo[0], yo[1], yo[2], yo[3]);
          }
        }
      }
    }
  }
  if (timed) trace[kUnitTimes + 3 * unit + 2] = globaltimer_ns();
}

// ================================================================ kernels
// split form, kernel 1: items j = blockIdx.x + k * gridDim.x < n_items,
// (chunk j / H, head j % H); two CTAs per SM
// (kSide: also the PrepSide copies)
template <bool kSide>
__global__ void __launch_bounds__(kPrepThreads, 2)
tc_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const float* __restrict__ alpha,
               const float* __restrict__ beta, SeqMap map, int32_t H,
               uint8_t* __restrict__ scratch, unsigned* status, uint64_t* __restrict__ trace,
               int64_t n_items, int32_t dv, ConvIn cv, PrepSide side) {
  extern __shared__ uint8_t smem_raw[];
  prep_role<false, kSide>(align_smem_1024(smem_raw), &tm_q, &tm_k, &tm_v, alpha, beta, map, H,
                          scratch, nullptr, status, dv, cv,
                          trace ? trace + kPrepTraceOffset : nullptr, trace, n_items, blockIdx.x,
                          gridDim.x, side);
}

// split form, kernel 2: one CTA per unit (blockIdx = sequence, head, 128-row
// slice of S)
__global__ void __launch_bounds__(kStateThreads, 1)
tc_state_kernel(const __grid_constant__ CUtensorMap tm_k, const float* __restrict__ S0,
                __nv_bfloat16* __restrict__ out, float* __restrict__ S_final, SeqMap map,
                int32_t H, const uint8_t* __restrict__ scratch, unsigned* status,
                uint64_t* __restrict__ trace, int32_t trace_chunks, int32_t dv,
                float* __restrict__ sdump, SegRoute route, NormGate ng) {
  extern __shared__ uint8_t smem_raw[];
  // a 1-D grid: the slice fastest (a head's units are neighbours, and the
  // pair of a cluster), then the head, then the unit's x in the route's order
  const int ns = dv / 128;
  const int lin = blockIdx.x, slice = lin % ns, h = (lin / ns) % H, rank = lin / (ns * H);
  const int x = route.order ? route.order[rank] : rank;
  const UnitRoute u = route_unit(route, S0, S_final, x, map.N, (int64_t)H * dv * kDK);
  // the whole CTA, before any barrier or TMEM allocation; an A chain has
  // dk rows
  if (!u.run || (u.ident && 128 * slice >= kDK)) return;
  state_role<false>(align_smem_1024(smem_raw), &tm_k, u.S0, u.write_out ? out : nullptr,
                    u.S_final, map, H, scratch, nullptr, status, trace, trace_chunks, dv,
                    x >= map.N ? x - map.N : x, h, slice, sdump, ng, u.ident);
}

// (fused form with the read-out, after a worker's prep items) Eq. 20 over
// the chunks' rows.  Each warp of each worker takes its own items in the
// prep's chunk-position order (item j = (worker * 8 + warp) + k * n_workers
// * 8), so that eight items per worker are in flight and no item waits
// behind another's flags: lane 0 waits (bounded) until both 128-row units of
// the item's head report the chunk's output rows out; then a lane takes
// the 16-byte column group `lane` of every row, eight rows at a time with
// all their loads in flight, the row's sum of squares (of the bf16 values
// stored) by a warp reduction, then the split form's arithmetic.  The state
// units thus add nothing to their chains.  dv = 256.
__device__ __forceinline__ void readout_role(const SeqMap& map, int32_t H, int32_t dv,
                                             const NormGate& ng, __nv_bfloat16* __restrict__ out,
                                             unsigned* status, int64_t n_items, int64_t worker,
                                             int64_t n_workers) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ns = dv / 128;
  float w8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w8[i] = __ldg(ng.w + 8 * lane + i);
  const float inv_dv = 1.f / (float)dv;
  const int64_t stride = n_workers * (kPrepThreads / 32);
  for (int64_t j = worker * (kPrepThreads / 32) + warp; j < n_items; j += stride) {
    PrepItem it;
    if (!prep_item<true>(map, H, j, it)) continue;
    int ok = 1;
    if (lane == 0) {
      const uint32_t* f = ng.flags + ((size_t)it.n * H + it.h) * ns;
      const uint32_t need = (uint32_t)(it.ci - map.chunk_begin(it.n) + 1);
      const uint64_t t_start = globaltimer_ns();
      for (int k = 0; k < ns && ok; ++k) {
        // a chunk of the chain takes a few microseconds: poll at about that
        // pace, so that hundreds of waiting warps do not crowd the L2 the
        // chains' loads go through
        while (ld_relaxed_gpu(f + k) < need) {
          if (globaltimer_ns() - t_start >= kReadyWaitNs) {
            ok = 0;
            break;
          }
          __nanosleep(2000);
        }
      }
      if (ok) fence_acq_rel_gpu();
      else flag_status(status, GDN_ERR_TIMEOUT);
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    for (int r0 = 0; r0 < it.L; r0 += 8) {
      uint4 ov[8], gv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (r0 + u < it.L) {
          const size_t row = (size_t)(it.t0 + r0 + u) * H + it.h;
          ov[u] = *reinterpret_cast<const uint4*>(out + row * dv + 8 * lane);
          gv[u] = __ldg(reinterpret_cast<const uint4*>(ng.gate + row * dv + 8 * lane));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (r0 + u < it.L) {   // uniform across the warp
          const uint32_t o4[4] = {ov[u].x, ov[u].y, ov[u].z, ov[u].w};
          const uint32_t g4[4] = {gv[u].x, gv[u].y, gv[u].z, gv[u].w};
          float ssum = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = bf16_lo(o4[e]), b = bf16_hi(o4[e]);
            ssum = fmaf(a, a, ssum);
            ssum = fmaf(b, b, ssum);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
          const float rs = rsqrtf(ssum * inv_dv + ng.eps);
          uint32_t yo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float g0 = bf16_lo(g4[e]), g1 = bf16_hi(g4[e]);
            const float a0 = ng.act == GDN_GATE_SIGMOID ? __fdividef(1.f, 1.f + __expf(-g0))
                                                        : __fdividef(g0, 1.f + __expf(-g0));
            const float a1 = ng.act == GDN_GATE_SIGMOID ? __fdividef(1.f, 1.f + __expf(-g1))
                                                        : __fdividef(g1, 1.f + __expf(-g1));
            yo[e] = pack_bf16(bf16_lo(o4[e]) * rs * w8[2 * e] * a0,
                              bf16_hi(o4[e]) * rs * w8[2 * e + 1] * a1);
          }
          const size_t row = (size_t)(it.t0 + r0 + u) * H + it.h;
          *reinterpret_cast<uint4*>(out + row * dv + 8 * lane) = make_uint4(yo[0], yo[1], yo[2], yo[3]);
        }
      }
    }
  }
}

// fused form: cooperative, one CTA per SM; CTAs [0, n_state) are the state
// units (with ns = dv / 128 slices of S per head, unit u = (sequence
// u / (ns H), head (u / ns) % H, slice u % ns)), the rest
// prep workers over all chunk positions in order; ready[] holds a flag per
// (chunk, head).  kNorm: the layer's read-out (Eq. 20) by the workers after
// their prep items; without it the state units get a NormGate known to be
// empty at compile time, so that no read-out code stays in their chains.
template <bool kNorm>
__global__ void __launch_bounds__(kStateThreads, 1)
tc_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kb,
                const float* __restrict__ alpha, const float* __restrict__ beta,
                const float* __restrict__ S0, __nv_bfloat16* __restrict__ out,
                float* __restrict__ S_final, SeqMap map, int32_t H, uint8_t* __restrict__ scratch,
                uint32_t* ready, unsigned* status, uint64_t* __restrict__ trace,
                int32_t trace_chunks, int32_t n_state, int32_t dv, float* __restrict__ sdump,
                ConvIn cv, NormGate ng) {
  static_assert(kPrepThreads == kStateThreads, "one block shape for both roles");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align_smem_1024(smem_raw);
  if ((int32_t)blockIdx.x < n_state) {
    const int u = blockIdx.x;
    const int ns = dv / 128, n = u / (ns * H);
    const int64_t per_seq = (int64_t)H * dv * kDK;
    // the state units only report their progress to the read-out (gate and
    // weight stay with the workers), so no read-out arithmetic is in their chains
    NormGate progress{};
    if (kNorm) progress.flags = ng.flags;
    state_role<true>(sm, &tm_kb, S0 ? S0 + n * per_seq : nullptr, out,
                     S_final ? S_final + n * per_seq : nullptr, map, H, scratch, ready, status,
                     trace, trace_chunks, dv, n, (u / ns) % H, u % ns, sdump, progress);
  } else {
    int64_t positions = map.chunks_per_seq;
    if (map.cu_seqlens) {
      positions = 0;
      for (int n = 0; n < map.N; ++n) {
        const int64_t c = map.chunk_end(n) - map.chunk_begin(n);
        positions = c > positions ? c : positions;
      }
    }
    prep_role<true>(sm, &tm_q, &tm_k, &tm_v, alpha, beta, map, H, scratch, ready, status, dv, cv,
                    trace ? trace + kPrepTraceOffset : nullptr, trace, positions * map.N * H,
                    blockIdx.x - n_state, gridDim.x - n_state);
    if (kNorm)   // the read-out norm of the chunks, behind the chains
      readout_role(map, H, dv, ng, out, status, positions * map.N * H, blockIdx.x - n_state,
                   gridDim.x - n_state);
  }
}

// ======================================================= reverse state pass
// The backward's reverse recurrence over the chunks of a sequence, on the
// tensor cores (bf16 I/O), mirroring the forward state pass.  For a chunk with
// end-state gradient dS' (dv x dk; this unit holds 128 of its rows):
//   dU^T = (dO^T P^) + (dS' K^T) diag(d)         [rows of dS x 64 tokens]
//   dS   = gamma_L dS' + dO^T Q^ - dU^T W          (the gradient carried back)
// with P^, Q^, W and the decay factors read from the forward's own operand
// images (the backward's forward re-run leaves them in scratch).  Per chunk:
// MMA-X  D_X = dS' K^T (A: the bf16 copy of dS' in TMEM, B: the K tile
//        K-major, N = 64, 16 K-steps);
// MMA-P  D_P = dO^T P^ (A: the dO tile MN-major, B: P^ read MN-major, N = 64);
// E1     dU^T = D_P + d D_X -> fp32 dU to scratch, -dU^T as a bf16 A operand
//        in TMEM over D_X;
// MMA-S  D_S = dO^T Q^ + (-dU^T) W, as four N = 64 blocks of dk (the image's
//        64-row blocks of W and Q^ are 16 KB apart), K = 64 tokens;
// E2     dS = gamma_L dS' + D_S in fp32 registers, bf16 copy back to TMEM.
// Before E2 the unit stores dS' (fp32) for the chunk gradients.  Tokens past
// the chunk's end contribute nothing: their d is 0 and their rows and
// columns of P^ are 0.
constexpr uint32_t kR_WQ = 0;         // 2 x 64 KB: the [W | Q^] images
constexpr uint32_t kR_KP = 131072;    // 40 KB: K tile (32 KB) | P^ (8 KB)
constexpr uint32_t kR_O = 172032;     // 2 x 16 KB: dO tiles (two 64-column blocks)
constexpr uint32_t kR_D = 204800;     // 2 x 512 B: decay blocks (d_r, then G_r)
constexpr uint32_t kR_T = 205824;     // 8 x 2560 B: per-warp transpose tiles (32 x 20 floats)
constexpr uint32_t kR_END = 226304;
constexpr uint32_t kRevSmemTc = kR_END + 1024;
constexpr uint32_t kR_TX = 0, kR_TP = 64, kR_TSA = 128, kR_TS = 256;   // TMEM columns

__global__ void __launch_bounds__(kStateThreads, 1)
tc_reverse_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_o,
                  SeqMap map, int32_t H, int32_t dv, const uint8_t* __restrict__ images,
                  const float* __restrict__ dS_final, float* __restrict__ dS0,
                  float* __restrict__ dSp, float* __restrict__ dUo, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align_smem_1024(smem_raw);
  const int ns = dv / 128;
  const int lin = blockIdx.x, slice = lin % ns, h = (lin / ns) % H, n = lin / (ns * H);
  __shared__ uint64_t bar_wq[2], bar_kp, bar_o[2], bar_m1, bar_m2;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, colhalf = warp >> 2;
  const uint32_t iloc = 32 * quarter + lane;
  const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
  const int64_t cb = map.chunk_begin(n), ce = map.chunk_end(n);
  const int64_t s_begin = map.seq_begin(n), s_end = map.seq_end(n);
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_wq[b], 1);
      mbar_init(&bar_o[b], 1);
    }
    mbar_init(&bar_kp, 1);
    mbar_init(&bar_m1, 1);
    mbar_init(&bar_m2, 1);
    fence_barrier_init();
    s_abort = 0;
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_o);
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  // this thread's 128 columns of row iloc of dS (fp32), from dS_final
  float S[128];
  const size_t srow = (((size_t)n * H + h) * dv + 128 * slice + iloc) * kDK + 128 * colhalf;
  if (dS_final) {
    const float4* p = reinterpret_cast<const float4*>(dS_final + srow);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float4 t = p[j];
      S[4 * j] = t.x; S[4 * j + 1] = t.y; S[4 * j + 2] = t.z; S[4 * j + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 128; ++j) S[j] = 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  auto store_operand = [&]() {   // bf16 copy of this thread's dS columns into TMEM
#pragma unroll
    for (int hq = 0; hq < 2; ++hq) {
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = pack_bf16(S[64 * hq + 2 * j], S[64 * hq + 2 * j + 1]);
      tmem_st32(tmem + lane_off + kR_TSA + 64 * colhalf + 32 * hq, r);
    }
    tmem_st_wait();
  };
  store_operand();
  // every warp's rows of the operand are in TMEM before the first MMA-X
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  auto img_of = [&](int64_t ci) { return images + (size_t)(ci * H + h) * img_stride(dv); };
  auto t0_of = [&](int64_t ci) { return (int32_t)(s_begin + (ci - cb) * kC); };
  // copies by single threads of warps 1-3, counted for a clean exit after a timeout
  constexpr int kLK = 32, kLW = 64, kLO = 96;
  uint32_t n_wq[2] = {0, 0}, n_kp = 0, n_o[2] = {0, 0};
  auto issue_kp = [&](int64_t ci) {   // the K tile and P^
    mbar_arrive_expect_tx(&bar_kp, 40960);
    tma_load_4d(sm + kR_KP, &tm_k, 0, t0_of(ci), 0, h, &bar_kp);
    tma_load_1d(sm + kR_KP + 32768, img_of(ci) + kImgP, 8192, &bar_kp);
    ++n_kp;
  };
  auto issue_o = [&](int64_t ci, int b) {   // this unit's dO columns and the decay block
    mbar_arrive_expect_tx(&bar_o[b], 16384 + 512);
    for (int bb = 0; bb < 2; ++bb)
      tma_load_3d(sm + kR_O + b * 16384 + bb * 8192, &tm_o, 128 * slice + 64 * bb, h, t0_of(ci),
                  &bar_o[b]);
    tma_load_1d(sm + kR_D + b * 512, img_of(ci) + kImgU0 + slice * kImgHalf + kImgDecay, 512,
                &bar_o[b]);
    ++n_o[b];
  };
  auto issue_wq = [&](int64_t ci, int b) {
    mbar_arrive_expect_tx(&bar_wq[b], 65536);
    tma_load_1d(sm + kR_WQ + b * 65536, img_of(ci) + kImgWQ, 65536, &bar_wq[b]);
    ++n_wq[b];
  };
  if (ce > cb) {
    if (tid == kLK) issue_kp(ce - 1);
    if (tid == kLO) issue_o(ce - 1, 0);
    if (tid == kLW) {
      issue_wq(ce - 1, 0);
      if (ce - 2 >= cb) issue_wq(ce - 2, 1);
    }
  }
  const size_t dsp_row = 128 * slice + iloc;
  for (int64_t ci = ce - 1; ci >= cb && !s_abort; --ci) {
    const int64_t it = ce - 1 - ci;
    const int b = (int)(it & 1);
    const uint32_t par = (uint32_t)(it & 1), bpar = (uint32_t)((it >> 1) & 1);
    const int64_t t0 = t0_of(ci);
    const int L = (int)min((int64_t)kC, s_end - t0);
    const size_t u = (size_t)(ci * H + h);
    const float* sD = reinterpret_cast<const float*>(sm + kR_D + b * 512);
    if (tid == kLO && ci - 1 >= cb) issue_o(ci - 1, b ^ 1);
    // MMA-X and MMA-P
    if (tid == 0) {
      if (!mbar_wait(&bar_kp, par) || !mbar_wait(&bar_o[b], bpar)) {
        s_abort = 1;
      } else {
        tc_fence_after();
        const uint32_t sK = smem_u32(sm + kR_KP), sP = sK + 32768;
        const uint32_t sO = smem_u32(sm + kR_O + b * 16384);
        const uint32_t idx = idesc_bf16(128, 64, 0, 0), idp = idesc_bf16(128, 64, 1, 1);
        for (int s = 0; s < 16; ++s)
          mma_bf16_ts(tmem + kR_TX, tmem + kR_TSA + 8 * s,
                      smem_desc(sK + (s >> 2) * 8192 + (s & 3) * 32, 16, 1024, kSwizzle128B), idx,
                      s > 0);
        for (int s = 0; s < 4; ++s)
          mma_bf16(tmem + kR_TP, smem_desc(sO + s * 2048, 8192, 1024, kSwizzle128B),
                   smem_desc(sP + s * 2048, 8192, 1024, kSwizzle128B), idp, s > 0);
        mma_commit(&bar_m1);
      }
    }
    // dS' of this chunk, for the chunk gradients.  A warp holds 32 rows.  In
    // the tiled layout (dv = 256) it is stored as bf16, as this pass's own
    // MMAs read dS, and a store of the warp covers 256 contiguous bytes;
    // row-major (fp32), each 16-byte piece would be its own L2 transaction, so
    // 16 columns at a time go through a per-warp tile in shared memory and
    // leave as four rows of 64 contiguous bytes per store.
    if (tiled_states(dv)) {   // lanes: consecutive rows
      uint2* p = reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(dSp) +
                                          u * dv * kDK) +
                 (size_t)32 * colhalf * dv + dsp_row;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        p[(size_t)j * dv] = make_uint2(pack_bf16(S[4 * j], S[4 * j + 1]),
                                       pack_bf16(S[4 * j + 2], S[4 * j + 3]));
    } else {
      float* tile = reinterpret_cast<float*>(sm + kR_T + warp * 2560);
      float* row0 = dSp + (u * dv + 128 * slice + 32 * quarter) * kDK + 128 * colhalf;
      const int rr = lane >> 2, c4 = lane & 3;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<float4*>(tile + lane * 20 + 4 * k) =
              make_float4(S[16 * q + 4 * k], S[16 * q + 4 * k + 1], S[16 * q + 4 * k + 2],
                          S[16 * q + 4 * k + 3]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 8 * i + rr;
          *reinterpret_cast<float4*>(row0 + (size_t)r * kDK + 16 * q + 4 * c4) =
              *reinterpret_cast<const float4*>(tile + r * 20 + 4 * c4);
        }
        __syncwarp();
      }
    }
    // E1: dU^T = D_P + d D_X
    if (!mbar_wait(&bar_m1, par)) {
      flag_status(status, GDN_ERR_TIMEOUT);
      s_abort = 1;
    } else {
      tc_fence_after();
      if (tid == kLK && ci - 1 >= cb) issue_kp(ci - 1);   // K / P^ are read
      uint32_t gx[32], gp[32];
      tmem_ld32(tmem + lane_off + kR_TX + 32 * colhalf, gx);
      tmem_ld32(tmem + lane_off + kR_TP + 32 * colhalf, gp);
      tmem_ld_wait();
      uint32_t pk[16];
      float* du_out = dUo + (u * kC + 32 * colhalf) * dv + dsp_row;
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const int r = 32 * colhalf + j;
        const float d0 = fmaf(sD[r], __uint_as_float(gx[j]), __uint_as_float(gp[j]));
        const float d1 = fmaf(sD[r + 1], __uint_as_float(gx[j + 1]), __uint_as_float(gp[j + 1]));
        du_out[(size_t)j * dv] = d0;
        du_out[(size_t)(j + 1) * dv] = d1;
        pk[j >> 1] = pack_bf16(-d0, -d1);
      }
      tmem_st16(tmem + lane_off + kR_TX + 32 * colhalf, pk);
      tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (s_abort) break;
    // MMA-S: D_S = dO^T Q^ + (-dU^T) W over four 64-column blocks of dk
    if (tid == 0) {
      if (!mbar_wait(&bar_wq[b], bpar)) {
        s_abort = 1;
      } else {
        tc_fence_after();
        const uint32_t sW = smem_u32(sm + kR_WQ + b * 65536);
        const uint32_t sO = smem_u32(sm + kR_O + b * 16384);
        const uint32_t idq = idesc_bf16(128, 64, 1, 0), idw = idesc_bf16(128, 64, 0, 0);
        for (int bk = 0; bk < 4; ++bk)
          for (int s = 0; s < 4; ++s)
            mma_bf16(tmem + kR_TS + 64 * bk, smem_desc(sO + s * 2048, 8192, 1024, kSwizzle128B),
                     smem_desc(sW + bk * 16384 + 8192 + s * 32, 16, 1024, kSwizzle128B), idq, s > 0);
        for (int bk = 0; bk < 4; ++bk)
          for (int s = 0; s < 4; ++s)
            mma_bf16_ts(tmem + kR_TS + 64 * bk, tmem + kR_TX + col_U(s),
                        smem_desc(sW + bk * 16384 + s * 32, 16, 1024, kSwizzle128B), idw, 1);
        mma_commit(&bar_m2);
      }
    }
    // E2: dS = gamma_L dS' + D_S, and its bf16 copy (MMA-X has read the old one)
    if (!mbar_wait(&bar_m2, par)) {
      flag_status(status, GDN_ERR_TIMEOUT);
      s_abort = 1;
    } else {
      tc_fence_after();
      if (tid == kLW && ci - 2 >= cb) issue_wq(ci - 2, b);   // this chunk's W | Q^ are read
      const float gC = exp_fast(sD[64 + L - 1]);
      const uint32_t tS = tmem + lane_off + kR_TS + 128 * colhalf;
      const uint32_t tA = tmem + lane_off + kR_TSA + 64 * colhalf;
      uint32_t g[2][16];
      tmem_ld16(tS, g[0]);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        tmem_ld_wait_regs(g[q & 1]);
        if (q + 1 < 8) tmem_ld16(tS + 16 * (q + 1), g[(q + 1) & 1]);
        uint32_t pk[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float s0 = fmaf(gC, S[16 * q + j], __uint_as_float(g[q & 1][j]));
          const float s1 = fmaf(gC, S[16 * q + j + 1], __uint_as_float(g[q & 1][j + 1]));
          S[16 * q + j] = s0;
          S[16 * q + j + 1] = s1;
          pk[j >> 1] = pack_bf16(s0, s1);
        }
        tmem_st8(tA + 8 * q, pk);
      }
      tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (!s_abort && dS0) {
    float4* p = reinterpret_cast<float4*>(dS0 + srow);
#pragma unroll
    for (int j = 0; j < 32; ++j) p[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
  }
  if (s_abort && (tid == kLK || tid == kLW || tid == kLO)) {   // let copies in flight land
    flag_status(status, GDN_ERR_TIMEOUT);
    const uint64_t lim = 100000000ull;
    for (int b = 0; b < 2; ++b) {
      if (tid == kLW && n_wq[b]) mbar_wait(&bar_wq[b], (n_wq[b] - 1) & 1, lim);
      if (tid == kLO && n_o[b]) mbar_wait(&bar_o[b], (n_o[b] - 1) & 1, lim);
    }
    if (tid == kLK && n_kp) mbar_wait(&bar_kp, (n_kp - 1) & 1, lim);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

constexpr uint32_t kPrepSmemSplit = PrepSmem<false>::BYTES;
constexpr uint32_t kFusedSmem = kStateSmem > PrepSmem<true>::BYTES ? kStateSmem : PrepSmem<true>::BYTES;
static_assert(PrepSmem<false>::A == 65536 && PrepSmem<true>::A % 1024 == 0, "prep layout");
// the fused form runs only if this many SMs are left for prep workers
constexpr int kMinPrepWorkers = 32;

// ------------------------------------------------------------- host side
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = (EncodeFn)p;
  }
  return fn;
}

// [T_total][H][D] bf16 viewed as (feature, head, token); box 64 x 1 x 64,
// 128-byte swizzle; token rows past the end of the tensor read as zero.
bool make_token_map(CUtensorMap* m, const void* base, int64_t T_total, int32_t H, int32_t D = kDK) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  memset(m, 0, sizeof *m);
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(T_total > 0 ? T_total : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same tensor viewed as (64 features, token, 4 feature blocks, head) so
// that one box of 64 x 64 x 4 x 1 lands the four 64-column blocks of a
// chunk's 64 tokens one after another: the MN-major image the state pass
// feeds to its MMA, in a single TMA copy.
bool make_token_map_blocked(CUtensorMap* m, const void* base, int64_t T_total, int32_t H) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  memset(m, 0, sizeof *m);
  cuuint64_t dims[4] = {64, (cuuint64_t)(T_total > 0 ? T_total : 1), 4, (cuuint64_t)H};
  cuuint64_t strides[3] = {(cuuint64_t)H * kDK * 2, 128, (cuuint64_t)kDK * 2};
  cuuint32_t box[4] = {64, 64, 4, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device launch facts, looked up once: SM count, and whether the fused
// form can be launched (cooperative launches supported and one fused CTA
// fits on an SM).
struct DeviceFacts {
  int sms = 0;
  bool fused_ok = false;
  bool ready = false;
};

DeviceFacts* device_facts() {
  static DeviceFacts facts[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  DeviceFacts& f = facts[dev];
  if (!f.ready) {
    int coop = 0, per_sm = 0, per_sm_norm = 0;
    if (cudaDeviceGetAttribute(&f.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
        cudaFuncSetAttribute(tc_prep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPrepSmemSplit) != cudaSuccess ||
        cudaFuncSetAttribute(tc_prep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPrepSmemSplit) != cudaSuccess ||
        cudaFuncSetAttribute(tc_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kStateSmem) != cudaSuccess ||
        cudaFuncSetAttribute(tc_fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kFusedSmem) != cudaSuccess ||
        cudaFuncSetAttribute(tc_fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kFusedSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_fused_kernel<false>,
                                                      kStateThreads, kFusedSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_norm, tc_fused_kernel<true>,
                                                      kStateThreads, kFusedSmem) != cudaSuccess)
      return nullptr;
    f.fused_ok = coop != 0 && per_sm >= 1 && per_sm_norm >= 1;
    f.ready = true;
  }
  return &f;
}

}  // namespace

// phase-timeline buffer for the state pass and, at kPrepTraceOffset, for the
// first prep worker (test hook; null when off)
uint64_t* g_trace = nullptr;
int32_t g_trace_chunks = 0;
int32_t g_last_tc_form = -1;

// operand images, then one ready flag per (chunk, head) for the fused form
size_t prefill_tc_scratch_bytes(int64_t max_chunks, int32_t H, int32_t dv) {
  const size_t items = (size_t)max_chunks * H;
  return items * img_stride(dv) + align_up(items * sizeof(uint32_t), 256);
}

size_t prefill_tc_image_stride() { return kImgStride; }

cudaError_t launch_prefill_tc(const PrefillLaunch& a, cudaStream_t stream, bool prep_only) {
  static_assert(kDK == 256, "image layouts assume dk = 256");
  const int32_t dv = a.dv;
  if (!supported_dv(dv)) return cudaErrorInvalidValue;
  const int64_t T_total = a.map.cu_seqlens ? a.map.T : (int64_t)a.map.N * a.map.T;
  CUtensorMap tq, tk, tv, tkb;
  if (a.cv.qkv) {
    // the packed projection as 3H heads of 256 channels a token (q | k | v),
    // and the state pass's keys from the prep's processed copy
    if (dv != kDK || !make_token_map(&tq, a.cv.qkv, T_total, 3 * a.H) ||
        !make_token_map_blocked(&tkb, a.cv.k_out, T_total, a.H))
      return cudaErrorInvalidValue;
    tk = tq;
    tv = tq;
  } else if (!make_token_map(&tq, a.q, T_total, a.H) || !make_token_map(&tk, a.k, T_total, a.H) ||
             !make_token_map(&tv, a.v, T_total, a.H, dv) ||
             !make_token_map_blocked(&tkb, a.k, T_total, a.H)) {
    return cudaErrorInvalidValue;
  }
  DeviceFacts* f = device_facts();
  if (!f) return cudaErrorUnknown;
  cudaError_t e;
  uint8_t* scr = (uint8_t*)a.scratch;
  const int64_t items = a.max_chunks * a.H;
  uint32_t* ready = (uint32_t*)(scr + (size_t)items * img_stride(dv));
  const int64_t n_state = (int64_t)a.map.N * a.H * (dv / 128);

  if (!prep_only && !a.state_only && a.allow_overlap && a.route.pass == 0 &&
      (!a.ng.gate || (a.ng.flags && dv == 256)) &&
      f->fused_ok && items > 0 &&
      n_state + kMinPrepWorkers <= f->sms) {
    if ((e = cudaMemsetAsync(ready, 0, (size_t)items * sizeof(uint32_t), stream)) != cudaSuccess)
      return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)f->sms);
    cfg.blockDim = dim3(kStateThreads);
    cfg.dynamicSmemBytes = kFusedSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, a.ng.gate ? tc_fused_kernel<true> : tc_fused_kernel<false>,
                           tq, tk, tv, tkb, a.alpha, a.beta, a.S0, (__nv_bfloat16*)a.out,
                           a.S_final, a.map, a.H, scr, ready, a.status, g_trace, g_trace_chunks,
                           (int32_t)n_state, dv, a.state_dump, a.cv, a.ng);
    if (e == cudaSuccess) {
      count_launches(1);
      g_last_tc_form = 1;
      return cudaSuccess;
    }
    // not all CTAs can be resident right now (e.g. SMs held by another
    // context): clear the launch error and take the split form
    if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    (void)cudaGetLastError();
  }

  if (items > 0 && !a.state_only) {
    const int64_t slots = 2 * (int64_t)f->sms;
    const unsigned grid = (unsigned)(items < slots ? items : slots);
    if (a.side.KK)
      tc_prep_kernel<true><<<grid, kPrepThreads, kPrepSmemSplit, stream>>>(
          tq, tk, tv, a.alpha, a.beta, a.map, a.H, scr, a.status, g_trace, items, dv, a.cv,
          a.side);
    else
      tc_prep_kernel<false><<<grid, kPrepThreads, kPrepSmemSplit, stream>>>(
          tq, tk, tv, a.alpha, a.beta, a.map, a.H, scr, a.status, g_trace, items, dv, a.cv,
          a.side);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (prep_only) return cudaSuccess;
  g_last_tc_form = 0;
  const int64_t n_blocks = (int64_t)a.map.N * (a.route.pass == 1 ? 2 : 1) * a.H * (dv / 128);
  if (n_blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)n_blocks);
  if (a.ng.gate) {
    // the read-out norm: the two units of a head form a cluster
    if (dv != 256) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kStateThreads);
    cfg.dynamicSmemBytes = kStateSmem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;   // the two slices of a head: neighbours in the grid
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, tc_state_kernel, tkb, a.S0, (__nv_bfloat16*)a.out, a.S_final,
                           a.map, a.H, (const uint8_t*)scr, a.status, g_trace, g_trace_chunks, dv,
                           a.state_dump, a.route, a.ng);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  tc_state_kernel<<<grid, kStateThreads, kStateSmem, stream>>>(
      tkb, a.S0, (__nv_bfloat16*)a.out, a.S_final, a.map, a.H, scr, a.status, g_trace,
      g_trace_chunks, dv, a.state_dump, a.route, a.ng);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_reverse_tc(const ReverseLaunch& r, cudaStream_t stream) {
  if (!supported_dv(r.dv)) return cudaErrorInvalidValue;
  const int64_t n_blocks = (int64_t)r.map.N * r.H * (r.dv / 128);
  if (n_blocks <= 0) return cudaSuccess;
  if (n_blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  CUtensorMap tk, to;
  if (!make_token_map_blocked(&tk, r.k, r.T_total, r.H) ||
      !make_token_map(&to, r.dout, r.T_total, r.H, r.dv))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_reverse_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kRevSmemTc);
  if (e != cudaSuccess) return e;
  tc_reverse_kernel<<<(unsigned)n_blocks, kStateThreads, kRevSmemTc, stream>>>(
      tk, to, r.map, r.H, r.dv, r.images, r.dS_final, r.dS0, r.dSp, r.dU, r.status);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace gdn
