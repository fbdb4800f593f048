// Fused batched beam-search step (sm_103a): two kernels per step.
//
// bs_stream_kernel, one CTA per SM: the R = B*W logit rows are cut into G equal
// ranges of the flattened [R, V] index space.  In each CTA a producer warp
// streams the range through a 6-stage ring of 32 KiB shared-memory chunks with
// bulk (TMA) copies completing on mbarriers, and 16 consumer warps read each
// chunk once from shared memory: per 32-element tile a thread updates an
// online log-sum-exp (log2 domain, SFU exp2) and compares the tile maximum
// with a CTA-wide threshold key.  Only a lane whose tile can hold one of the
// row's 2W best (logit, token) pairs leaves the streaming loop, to queue the
// qualifying keys in a CTA-wide shared-memory queue.  The threshold is seeded
// at the start of every row segment from the consumers' first-tile maxima and
// is raised from the queue every 16 pushes; it never passes the segment's K-th
// best, so an element below it is provably outside the row's top K.  A row
// segment ends in one partial (max, scaled sum, K sorted keys).
//
// bs_merge_kernel, one CTA per sentence, launched as a programmatic dependent
// of the stream kernel (it starts as the stream CTAs retire and waits for
// their writes): each row's LSE and top-K from its partials, the sentence's
// best 2W candidates by (score desc, flat index asc) found by ranking, the
// walk that moves EOS hits into the finished set, the stopping test, the
// outputs and the in-place sequence gather.  No CTA waits on another CTA of
// its own grid; every mbarrier wait is bounded.
//
// What is computed follows "Transformers中的Beam Search高效实现" (section
// 多个样本同时进行beam search: log_softmax, add beam_scores, view [batch, W*V],
// top-k, beam_id = j // V, token_id = j % V, BeamHypotheses.add / is_done, pad
// rows of finished sentences) and "9.2 贪心搜索与束搜索" (§9.2.2 four sub-steps,
// "何时结束" early_stopping modes; §9.2.3 length penalty).

#include <cfloat>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "bs_internal.h"

namespace vbs {

constexpr int BS_NC = 512;                        // consumer threads
constexpr int BS_NCW = BS_NC / 32;                // consumer warps
constexpr int BS_NT = BS_NC + 32;                 // + the producer warp
constexpr int BS_NW = BS_NT / 32;
constexpr int BS_U = 4;                           // 16-byte vectors per consumer per chunk
constexpr int STAGE_BYTES = BS_NC * BS_U * 16;    // 32 KiB
constexpr int NSTAGE = 6;
constexpr int QCAP = 1024;                        // the CTA's candidate queue (one row segment)
constexpr int QREFRESH = 16;                      // threshold refresh every QREFRESH pushes ...
constexpr int QREFRESH_MAX = 128;                 // ... while the queue holds at most this many
constexpr int SEQ_TILE_INTS = 2048;               // sequence gather tile (all W rows)
constexpr int BAR_CONSUMERS = 1;                  // named barrier of the consumer warps
constexpr int MG_NT = 256;                        // merge kernel threads
constexpr int MG_NW = MG_NT / 32;

// Merge (M, l) pairs in the log2 domain: sum = l * 2^M.
__device__ __forceinline__ void lse_merge(float& M, float& l, float M2, float l2) {
  const float Mn = fmaxf(M, M2);
  if (Mn == -INFINITY) { M = Mn; l = 0.f; return; }
  l = l * ex2(M - Mn) + l2 * ex2(M2 - Mn);
  M = Mn;
}

// ---------------------------------------------------------------------------------------
// selection helpers (one warp)
// ---------------------------------------------------------------------------------------

// K best of n keys by repeated warp max (destroys the keys; for large n).
__device__ void warp_select_topk(u64* keys, int n, int K, u64* out, int lane) {
  for (int round = 0; round < K; ++round) {
    u64 best = 0;
    int bi = -1;
    for (int c = lane; c < n; c += 32) {
      const u64 k = keys[c];
      if (k > best) { best = k; bi = c; }
    }
    const u64 g = warp_max_u64(best);
    if (bi >= 0 && best == g && g != 0) keys[bi] = 0;
    if (lane == 0) out[round] = g;
    __syncwarp();
  }
}

// K best of n unsorted keys by counting ranks (small n; keys unique, 0 = empty).
__device__ void warp_rank_topk(const u64* keys, int n, int K, u64* out, int lane) {
  if (lane < K) out[lane] = 0;
  __syncwarp();
  for (int j = lane; j < n; j += 32) {
    const u64 k = keys[j];
    if (k == 0) continue;
    int rank = 0;
    for (int q = 0; q < n; ++q) rank += keys[q] > k;
    if (rank < K) out[rank] = k;
  }
  __syncwarp();
}

// Number of entries of a descending list L[0..len) greater than k.
__device__ __forceinline__ int count_gt(const u64* L, int len, u64 k) {
  int lo = 0, hi = len;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (L[mid] > k) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// K best of nl descending lists of K keys each, by rank (binary search in the others).
__device__ void warp_merge_sorted(const u64* lists, int nl, int K, u64* out, int lane) {
  if (lane < K) out[lane] = 0;
  __syncwarp();
  for (int f = lane; f < nl * K; f += 32) {
    const int c = f / K, i = f - c * K;
    const u64 k = lists[f];
    if (k == 0) continue;
    int rank = i;
    for (int c2 = 0; c2 < nl && rank < K; ++c2)
      if (c2 != c) rank += count_gt(lists + c2 * K, K, k);
    if (rank < K) out[rank] = k;
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------------------
// shared memory
// ---------------------------------------------------------------------------------------

struct BsShared {                              // the stream kernel
  unsigned char ring[NSTAGE][STAGE_BYTES];     // the streamed chunks
  u64 q[QCAP];                                 // candidate keys of the current row segment
  u64 lbk[BS_NC];                              // first-tile lower bounds (threshold seed)
  u64 pool[64];
  u64 ptop[KMAX];                              // a partial's top K
  u64 full[NSTAGE], empty[NSTAGE];
  u64 thr;                                     // CTA threshold key
  int qcnt, ovf;
  float M[BS_NCW], l[BS_NCW];
};

struct MergeShared {                           // the merge kernel
  u64 rowscratch[WMAX * PART_KEYS];            // the rows' partial lists
  u64 wtop[WMAX * KMAX];                       // the W rows' sorted lists
  float candv[WMAX * KMAX];                    // their candidate scores, list order
  int nval[WMAX];
  int sel_w[KMAX], sel_i[KMAX];                // the sentence's best 2W, in order
  float sel_c[KMAX];
  int tile[SEQ_TILE_INTS];                     // the parents' sequence rows
  float s[WMAX];
  double f_ns[WMAX];
  int f_len[WMAX], f_serial[WMAX], f_src[WMAX];
  int f_count, f_next;
  double f_worst;
  float nb_score[WMAX];
  int nb_tok[WMAX], nb_row[WMAX];
  int done_now;
};

// ---------------------------------------------------------------------------------------
// the candidate queue
// ---------------------------------------------------------------------------------------

// Queue one key; true when the push completes a block of QREFRESH pushes.
__device__ __forceinline__ bool queue_push(BsShared& sh, u64 key) {
  const int pos = atomicAdd(&sh.qcnt, 1);
  if (pos < QCAP) sh.q[pos] = key;
  else sh.ovf = 1;
  return (pos % QREFRESH) == QREFRESH - 1;
}

// Warp-wide: raise the CTA threshold to a key with K-1 queued keys above it.  Other
// warps may be appending meanwhile: an entry not written yet reads 0 and is ignored,
// and a key seen with K-1 larger keys always has K queued keys at or above it, so the
// threshold never passes the segment's K-th best.
__device__ __noinline__ void queue_refresh(BsShared& sh, int K, int lane) {
  const volatile u64* vq = sh.q;
  const int n = min(*reinterpret_cast<volatile int*>(&sh.qcnt), QCAP);
  if (n < K || n > QREFRESH_MAX) return;
  for (int j = lane; j < n; j += 32) {
    const u64 k = vq[j];
    if (k == 0) continue;
    int rank = 0;
    for (int i = 0; i < n; ++i) rank += vq[i] > k;
    if (rank == K - 1) atomicMax(&sh.thr, k);
  }
}

// ---------------------------------------------------------------------------------------
// pass 1
// ---------------------------------------------------------------------------------------

struct Chunk {
  int r;
  int v0, len;              // elements of row r: [v0, v0 + len)
  bool first, last;         // first / last chunk of a row segment
};

// Walks a CTA's range [e0, e1) of the flattened [R, V] space in chunks of at most
// SE elements that never cross a row; one division at the start, none per chunk.
struct ChunkCursor {
  int r, r_last;
  int v, v_end_last, V, SE;
  bool fresh;
  __device__ __forceinline__ ChunkCursor(int64_t e0, int64_t e1, int V_, int SE_) : V(V_), SE(SE_), fresh(true) {
    r = static_cast<int>(e0 / V_);
    v = static_cast<int>(e0 - static_cast<int64_t>(r) * V_);
    r_last = static_cast<int>((e1 - 1) / V_);
    v_end_last = static_cast<int>(e1 - static_cast<int64_t>(r_last) * V_);
  }
  __device__ __forceinline__ bool more() const { return r <= r_last; }
  __device__ __forceinline__ Chunk next() {
    Chunk c;
    c.r = r;
    c.v0 = v;
    const int seg_end = r == r_last ? v_end_last : V;
    c.len = min(SE, seg_end - v);
    c.first = fresh;
    c.last = v + c.len == seg_end;
    v += c.len;
    fresh = c.last;
    if (c.last) { ++r; v = 0; }
    return c;
  }
};

__device__ __forceinline__ bool row_skipped(const BsArgs& a, int r) {
  return a.done[r / a.W] != 0 || a.scores[r] == -INFINITY;
}

// The producer: one lane keeps the ring full with bulk copies.
template <typename T>
__device__ void produce(const BsArgs& a, BsShared& sh, int64_t e0, int64_t e1) {
  constexpr int VEC = Vec16<T>::N;
  constexpr int64_t SE = static_cast<int64_t>(BS_NC) * BS_U * VEC;
  bool skip = false;
  ChunkCursor cur(e0, e1, a.V, static_cast<int>(SE));
  for (int c = 0; cur.more(); ++c) {
    const Chunk ch = cur.next();
    if (ch.first) skip = row_skipped(a, ch.r);
    const int slot = c % NSTAGE;
    if (c >= NSTAGE && !mbar_wait(&sh.empty[slot], static_cast<u32>(((c / NSTAGE) + 1) & 1)))
      set_status(a.status, VBS_ETIMEOUT);
    const u32 bytes = skip ? 0u : static_cast<u32>(ch.len * Elem<T>::BYTES);
    mbar_expect_tx(&sh.full[slot], bytes);
    if (bytes) {
      const char* src = reinterpret_cast<const char*>(a.logits) +
                        (static_cast<int64_t>(ch.r) * a.ld + ch.v0) * Elem<T>::BYTES;
      bulk_g2s(sh.ring[slot], src, bytes, &sh.full[slot]);
    }
  }
}

// Consumers, after a queue overflow: collect every key of the segment at or above
// the K-th best queued so far, re-reading the segment from global memory, until one
// pass fits in the queue.  Only adversarial orderings (e.g. ascending logits) get here.
template <typename T>
__device__ void rescan_segment(const BsArgs& a, BsShared& sh, int r, int64_t sv0, int64_t sv1) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  const char* row = reinterpret_cast<const char*>(a.logits) + static_cast<int64_t>(r) * a.ld * Elem<T>::BYTES;
  for (;;) {
    if (warp == 0) {
      warp_select_topk(sh.q, QCAP, K, sh.ptop, lane);
      if (lane == 0) { sh.thr = sh.ptop[K - 1]; sh.qcnt = 0; sh.ovf = 0; }
    }
    named_sync(BAR_CONSUMERS, BS_NC);
    for (int i = tid; i < QCAP; i += BS_NC) sh.q[i] = 0ull;
    const u64 thr = sh.thr;
    named_sync(BAR_CONSUMERS, BS_NC);
    for (int64_t v = sv0 + tid; v < sv1; v += BS_NC) {
      const u64 k = make_key(Elem<T>::load(row, v), static_cast<u32>(v));
      if (k >= thr) queue_push(sh, k);
    }
    named_sync(BAR_CONSUMERS, BS_NC);
    if (!sh.ovf) return;
    named_sync(BAR_CONSUMERS, BS_NC);
  }
}

// One lane's slow path: queue every element of its tile whose key reaches the
// threshold.  Out of line, so the streaming loop stays small; the tile comes packed.
template <typename T, int VEC>
__device__ __noinline__ bool push_tile(BsShared& sh, uint4 q0, uint4 q1, uint4 q2, uint4 q3, u32 okmask, u32 vb,
                                       float thr_x, u64 thr) {
  bool crossed = false;
  const uint4 qs[BS_U] = {q0, q1, q2, q3};
#pragma unroll
  for (int u = 0; u < BS_U; ++u) {
    if (!(okmask & (1u << u))) continue;
    float x[VEC];
    if constexpr (VEC == 1) x[0] = __uint_as_float(qs[u].x);
    else Vec16<T>::unpack(qs[u], x);
    const u32 vu = vb + static_cast<u32>(u * BS_NC * VEC);
#pragma unroll
    for (int e2 = 0; e2 < VEC; ++e2) {
      if (x[e2] >= thr_x) {
        const u64 k = make_key(x[e2], vu + e2);
        if (k >= thr) crossed |= queue_push(sh, k);
      }
    }
  }
  return crossed;
}

// The consumers: every chunk of the range, one row segment after the other.
template <typename T, bool TMA>
__device__ void consume(const BsArgs& a, BsShared& sh, int64_t e0, int64_t e1) {
  constexpr int VEC = TMA ? Vec16<T>::N : 1;
  constexpr int64_t SE = static_cast<int64_t>(BS_NC) * BS_U * VEC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  u64 thr = 0;
  float M = -INFINITY, m = -INFINITY, l = 0.f;
  bool skip = false;
  int seg_v0 = 0;
  ChunkCursor cur(e0, e1, a.V, static_cast<int>(SE));
  for (int c = 0; cur.more(); ++c) {
    const Chunk ch = cur.next();
    if (ch.first) {
      skip = row_skipped(a, ch.r);
      seg_v0 = ch.v0;
      thr = 0;
      M = -INFINITY;
      m = -INFINITY;
      l = 0.f;
    }
    const int n = ch.len / VEC;                     // vectors in this chunk
    uint4 q[BS_U];
    float xs[BS_U];
    bool ok[BS_U];
    if constexpr (TMA) {
      const int slot = c % NSTAGE;
      if (!mbar_wait(&sh.full[slot], static_cast<u32>((c / NSTAGE) & 1))) set_status(a.status, VBS_ETIMEOUT);
#pragma unroll
      for (int u = 0; u < BS_U; ++u) {
        const int i = tid + u * BS_NC;
        ok[u] = !skip && i < n;
        constexpr u32 NEG = VecMax<T>::NEG;
        q[u] = ok[u] ? *reinterpret_cast<const uint4*>(sh.ring[slot] + i * 16) : make_uint4(NEG, NEG, NEG, NEG);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[slot]);  // the slot may refill once every warp has its data
    } else {
      const char* row = reinterpret_cast<const char*>(a.logits) +
                        (static_cast<int64_t>(ch.r) * a.ld + ch.v0) * Elem<T>::BYTES;
#pragma unroll
      for (int u = 0; u < BS_U; ++u) {
        const int i = tid + u * BS_NC;
        ok[u] = !skip && i < n;
        xs[u] = ok[u] ? Elem<T>::load(row, i) : -INFINITY;
      }
    }
    if (!skip) {
      float tm;
      if constexpr (TMA) {
        u32 acc = VecMax<T>::NEG;
#pragma unroll
        for (int u = 0; u < BS_U; ++u) acc = VecMax<T>::fold(q[u], acc);
        tm = VecMax<T>::finish(acc);
      } else {
        tm = xs[0];
#pragma unroll
        for (int u = 1; u < BS_U; ++u) tm = fmaxf(tm, xs[u]);
      }
      // online log-sum-exp in the log2 domain: l = sum 2^(x*log2e - M)
      if (tm > m) {
        const float Mn = tm * LOG2E_F;
        l *= ex2(M - Mn);
        M = Mn;
        m = tm;
      }
      if (tm > -INFINITY) {
        float acc[BS_U];
#pragma unroll
        for (int u = 0; u < BS_U; ++u) {
          float x[VEC];
          if constexpr (TMA) Vec16<T>::unpack(q[u], x);
          else x[0] = xs[u];
#pragma unroll
          for (int e2 = 0; e2 < VEC; ++e2) x[e2] = ex2(fmaf(x[e2], LOG2E_F, -M));
#pragma unroll
          for (int w = 1; w < VEC; w <<= 1)
#pragma unroll
            for (int e2 = 0; e2 + w < VEC; e2 += 2 * w) x[e2] += x[e2 + w];
          acc[u] = x[0];
        }
#pragma unroll
        for (int w = 1; w < BS_U; w <<= 1)
#pragma unroll
          for (int u = 0; u + w < BS_U; u += 2 * w) acc[u] += acc[u + w];
        l += acc[0];
      }
      if (ch.first) {
        // the threshold seed: each warp offers its kw best first-tile lower bounds; the
        // K-th best of that pool is a lower bound of the segment's K-th best
        int ulast = -1;
#pragma unroll
        for (int u = 0; u < BS_U; ++u) ulast = ok[u] ? u : ulast;
        const u64 lb = ulast >= 0 ? make_key(tm, static_cast<u32>(ch.v0 + (tid + ulast * BS_NC) * VEC + VEC - 1))
                                  : 0ull;
        const int kw = max(2, (2 * K + BS_NCW - 1) / BS_NCW);
        sh.lbk[tid] = lb;
        for (int i = tid; i < QCAP; i += BS_NC) sh.q[i] = 0ull;
        if (tid == 0) { sh.qcnt = 0; sh.ovf = 0; }
        if (lane < kw) sh.pool[warp * kw + lane] = 0ull;
        __syncwarp();
        int rk = 0;
        for (int q2 = 0; q2 < 32; ++q2) rk += sh.lbk[warp * 32 + q2] > lb;
        if (lb != 0 && rk < kw) sh.pool[warp * kw + rk] = lb;
        named_sync(BAR_CONSUMERS, BS_NC);
        if (warp == 0) {
          const int np = BS_NCW * kw;
          u64 mine = 0;
          for (int j = lane; j < np; j += 32) {
            const u64 k = sh.pool[j];
            int rank = 0;
            for (int q2 = 0; q2 < np; ++q2) rank += sh.pool[q2] > k;
            if (k != 0 && rank == K - 1) mine = k;
          }
          const u64 seed = warp_max_u64(mine);      // 0 when fewer than K lower bounds exist
          if (lane == 0) sh.thr = seed;
        }
        named_sync(BAR_CONSUMERS, BS_NC);
        thr = sh.thr;
      } else {
        const u64 t2 = *reinterpret_cast<volatile u64*>(&sh.thr);
        thr = t2 > thr ? t2 : thr;
      }
      // candidates: only lanes whose tile can beat the threshold, one queue push per key
      const float thr_x = thr ? key_x(thr) : -INFINITY;
      bool crossed = false;
      if (tm >= thr_x && tm > -INFINITY) {
        u32 okmask = 0;
#pragma unroll
        for (int u = 0; u < BS_U; ++u) okmask |= ok[u] ? 1u << u : 0u;
        const u32 vb = static_cast<u32>(ch.v0 + tid * VEC);
        if constexpr (TMA) {
          crossed = push_tile<T, VEC>(sh, q[0], q[1], q[2], q[3], okmask, vb, thr_x, thr);
        } else {
          crossed = push_tile<T, 1>(sh, make_uint4(__float_as_uint(xs[0]), 0, 0, 0),
                                    make_uint4(__float_as_uint(xs[1]), 0, 0, 0),
                                    make_uint4(__float_as_uint(xs[2]), 0, 0, 0),
                                    make_uint4(__float_as_uint(xs[3]), 0, 0, 0), okmask, vb, thr_x, thr);
        }
      }
      if (__any_sync(FULL, crossed)) queue_refresh(sh, K, lane);
    }
    if (ch.last) {
      // ---- the segment's partial: (max, scaled sum, K sorted keys) ----
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float M2 = __shfl_xor_sync(FULL, M, off);
        const float l2 = __shfl_xor_sync(FULL, l, off);
        lse_merge(M, l, M2, l2);
      }
      if (lane == 0) { sh.M[warp] = M; sh.l[warp] = l; }
      named_sync(BAR_CONSUMERS, BS_NC);
      if (!skip && sh.ovf) rescan_segment<T>(a, sh, ch.r, seg_v0, static_cast<int64_t>(ch.v0) + ch.len);
      if (warp == 0) {
        float Mw = lane < BS_NCW ? sh.M[lane] : -INFINITY;
        float lw = lane < BS_NCW ? sh.l[lane] : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float M2 = __shfl_xor_sync(FULL, Mw, off);
          const float l2 = __shfl_xor_sync(FULL, lw, off);
          lse_merge(Mw, lw, M2, l2);
        }
        const int nq = skip ? 0 : min(sh.qcnt, QCAP);
        if (nq <= 128) warp_rank_topk(sh.q, nq, K, sh.ptop, lane);
        else warp_select_topk(sh.q, nq, K, sh.ptop, lane);
        const int pidx = static_cast<int>(blockIdx.x) - a.row_p0[ch.r];
        const int64_t slot = static_cast<int64_t>(ch.r) * a.P + pidx;
        if (lane < K) a.part_key[slot * K + lane] = sh.ptop[lane];
        if (lane == 0) { a.part_M[slot] = Mw; a.part_l[slot] = lw; }
      }
      named_sync(BAR_CONSUMERS, BS_NC);
    }
  }
}

// ---------------------------------------------------------------------------------------
// the stream kernel
// ---------------------------------------------------------------------------------------

template <typename T, bool TMA>
__global__ void __launch_bounds__(BS_NT, 1) bs_stream_kernel(const BsArgs a) {
  extern __shared__ __align__(128) unsigned char bs_smem[];
  BsShared& sh = *reinterpret_cast<BsShared*>(bs_smem);
  const int64_t total = static_cast<int64_t>(a.R) * a.V;
  const int64_t e0 = static_cast<int64_t>(blockIdx.x) * a.per;
  const int64_t e1 = min(e0 + a.per, total);
  if (e0 < e1) {
    if (threadIdx.x == 0) {
      for (int s = 0; s < NSTAGE; ++s) {
        mbar_init(&sh.full[s], 1);
        mbar_init(&sh.empty[s], BS_NCW);
      }
      fence_mbar_init();
    }
    __syncthreads();
    if ((threadIdx.x >> 5) == BS_NCW) {
      if constexpr (TMA) {
        if ((threadIdx.x & 31) == 0) produce<T>(a, sh, e0, e1);
      }
    } else {
      consume<T, TMA>(a, sh, e0, e1);
    }
  }
  // the merge grid may start filling the SMs this CTA leaves
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------------------
// the merge kernel: one CTA per sentence
// ---------------------------------------------------------------------------------------

// Warp-wide: row r's LSE (split hi + lo in fp32) and its sorted top-K list with scores.
__device__ void row_merge(const BsArgs& a, MergeShared& sm, int r, int w, int lane) {
  const int K = a.K;
  const float s = __ldcg(a.scores + r);
  if (s == -INFINITY) {
    // every candidate of the row is -inf: they rank by token id
    const int nv = K < a.V ? K : a.V;
    if (lane < K) {
      sm.wtop[w * K + lane] = lane < nv ? make_key(-INFINITY, static_cast<u32>(lane)) : 0ull;
      sm.candv[w * K + lane] = -INFINITY;
    }
    if (lane == 0) sm.nval[w] = nv;
    return;
  }
  const int n = a.row_np[r];
  const int64_t base = static_cast<int64_t>(r) * a.P;
  u64* scratch = sm.rowscratch + w * PART_KEYS;
  for (int c = lane; c < n * K; c += 32) scratch[c] = __ldcg(a.part_key + base * K + c);
  float Mc = -INFINITY, lc = 0.f;
  for (int c = lane; c < n; c += 32) lse_merge(Mc, lc, __ldcg(a.part_M + base + c), __ldcg(a.part_l + base + c));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float M2 = __shfl_xor_sync(FULL, Mc, off);
    const float l2 = __shfl_xor_sync(FULL, lc, off);
    lse_merge(Mc, lc, M2, l2);
  }
  __syncwarp();
  u64* out = sm.wtop + w * K;
  warp_merge_sorted(scratch, n, K, out, lane);
  const double lse = LN2_D * (static_cast<double>(Mc) + static_cast<double>(log2f(lc)));
  const float hi = static_cast<float>(lse);
  const float lo = static_cast<float>(lse - static_cast<double>(hi));
  if (lane == 0 && !(lse > -INFINITY && lse < INFINITY)) set_status(a.status, VBS_EINPUT);  // no finite logit, NaN, +inf
  if (lane < K) {
    const u64 k = out[lane];
    const float x = key_x(k);
    sm.candv[w * K + lane] = (k == 0 || x == -INFINITY) ? -INFINITY : s + ((x - hi) - lo);
  }
  const u32 nz = __ballot_sync(FULL, lane < K && out[lane] != 0);
  if (lane == 0) sm.nval[w] = __popc(nz);
}

// Entries of row w2 that rank before a candidate of score c from row w (w2 != w):
// a higher score, or the same score in a lower row.  Row lists are non-increasing.
__device__ __forceinline__ int count_better(const float* cv, int len, float c, bool lower_row) {
  int lo = 0, hi = len;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const float v = cv[mid];
    if (v > c || (lower_row && v == c)) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(MG_NT) bs_merge_kernel(const BsArgs a) {
  extern __shared__ __align__(16) unsigned char mg_smem[];
  MergeShared& sm = *reinterpret_cast<MergeShared*>(mg_smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int W = a.W, K = a.K;
  const int r0 = b * W;
  const int t = a.t;
  const int ld = a.seq_ld;
  const int TW = SEQ_TILE_INTS / W;            // columns per row in one gather tile
  const int nc0 = min(t, TW);

  // everything below reads what the stream kernel wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const bool was_done = a.done[b] != 0;

  if (!was_done) {
    // the first gather tile and the sentence state load while the rows merge
    for (int i = tid; i < W * nc0; i += MG_NT) {
      const int w = i / nc0, c = i - w * nc0;
      sm.tile[w * TW + c] = a.seqs[static_cast<int64_t>(r0 + w) * ld + c];
    }
    if (tid < W) {
      sm.s[tid] = a.scores[r0 + tid];
      sm.f_ns[tid] = a.fin_ns[r0 + tid];
      sm.f_len[tid] = a.fin_len[r0 + tid];
      sm.f_serial[tid] = a.fin_serial[r0 + tid];
      sm.f_src[tid] = -1;
    }
    if (tid == 0) {
      sm.f_count = a.fin_count[b];
      sm.f_next = a.fin_next[b];
      sm.f_worst = a.fin_worst[b];
    }
    for (int w = warp; w < W; w += MG_NW) row_merge(a, sm, r0 + w, w, lane);
  }
  __syncthreads();

  if (!was_done) {
    // rank every candidate of the W lists; the best 2W land in order
    for (int f = tid; f < W * K; f += MG_NT) {
      const int w = f / K, i = f - w * K;
      if (i >= sm.nval[w]) continue;
      const float c = sm.candv[f];
      int rank = i;
      for (int w2 = 0; w2 < W && rank < 2 * W; ++w2)
        if (w2 != w) rank += count_better(sm.candv + w2 * K, sm.nval[w2], c, w2 < w);
      if (rank < 2 * W) {
        sm.sel_w[rank] = w;
        sm.sel_i[rank] = i;
        sm.sel_c[rank] = c;
      }
    }
  }
  __syncthreads();

  if (tid == 0 && !was_done) {
    // the walk of the ranked candidates
    int new_cnt = 0;
    const float lp_t = static_cast<float>(a.lp_t);
    for (int rank = 0; rank < 2 * W && new_cnt < W; ++rank) {
      const int w = sm.sel_w[rank];
      const float c = sm.sel_c[rank];
      const u32 v = key_v(sm.wtop[w * K + sm.sel_i[rank]]);
      const int parent = r0 + w;
      if (a.eos >= 0 && static_cast<int>(v) == a.eos) {
        if (rank < W) {
          // BeamHypotheses.add(hyp = the parent's sequence, sum = c), |y| = t
          const double ns = static_cast<double>(c / lp_t);
          int slot = -1;
          if (sm.f_count < W) {
            slot = sm.f_count++;
            sm.f_worst = fmin(ns, sm.f_worst);
          } else if (ns > sm.f_worst) {
            slot = 0;                          // evict the worst; ties: the earliest inserted
            for (int q = 1; q < W; ++q)
              if (sm.f_ns[q] < sm.f_ns[slot] || (sm.f_ns[q] == sm.f_ns[slot] && sm.f_serial[q] < sm.f_serial[slot]))
                slot = q;
          }
          if (slot >= 0) {
            sm.f_ns[slot] = ns;
            sm.f_len[slot] = t;
            sm.f_serial[slot] = sm.f_next++;
            sm.f_src[slot] = parent;
            if (sm.f_count >= W) {
              double wmin = sm.f_ns[0];
              for (int q = 1; q < W; ++q) wmin = fmin(wmin, sm.f_ns[q]);
              sm.f_worst = wmin;
            }
          }
        }
      } else {
        sm.nb_score[new_cnt] = c;
        sm.nb_tok[new_cnt] = static_cast<int>(v);
        sm.nb_row[new_cnt] = parent;
        ++new_cnt;
      }
    }
    if (new_cnt < W) set_status(a.status, VBS_EINPUT);
    for (int q = new_cnt; q < W; ++q) { sm.nb_score[q] = -INFINITY; sm.nb_tok[q] = a.pad; sm.nb_row[q] = r0; }
    bool done = false;
    if (sm.f_count >= W)
      done = a.early_stopping == VBS_ES_TRUE ||
             sm.f_worst >= static_cast<double>(sm.sel_c[0]) / a.lp_bound;
    sm.done_now = done ? 1 : 0;
  }
  if (tid == 0 && was_done) sm.done_now = 1;
  __syncthreads();

  // the step's finished-sentence count: one atomic per sentence, issued before the writes
  unsigned old_cnt = 0;
  if (tid == 0) old_cnt = atomicAdd(reinterpret_cast<unsigned*>(a.done_count), (1u << 16) | sm.done_now);

  if (was_done) {
    if (tid < W) {
      a.beam_idx[r0 + tid] = -1;
      a.tokens[r0 + tid] = a.pad;
      a.scores[r0 + tid] = 0.f;
      a.seqs[static_cast<int64_t>(r0 + tid) * ld + t] = a.pad;
    }
  } else {
    if (tid < W) {
      a.beam_idx[r0 + tid] = sm.nb_row[tid];
      a.tokens[r0 + tid] = sm.nb_tok[tid];
      a.scores[r0 + tid] = sm.nb_score[tid];
      a.fin_ns[r0 + tid] = sm.f_ns[tid];
      a.fin_len[r0 + tid] = sm.f_len[tid];
      a.fin_serial[r0 + tid] = sm.f_serial[tid];
    }
    if (tid == 0) {
      a.fin_count[b] = sm.f_count;
      a.fin_next[b] = sm.f_next;
      a.fin_worst[b] = sm.f_worst;
      a.done[b] = sm.done_now;
    }
    // sequences: gather the parents' columns [0, t) in place (tile 0 is prefetched), append the token
    for (int c0 = 0; c0 < t; c0 += TW) {
      const int nc = min(TW, t - c0);
      if (c0 > 0) {
        __syncthreads();
        for (int i = tid; i < W * nc; i += MG_NT) {
          const int w = i / nc, c = i - w * nc;
          sm.tile[w * TW + c] = a.seqs[static_cast<int64_t>(r0 + w) * ld + c0 + c];
        }
        __syncthreads();
      }
      for (int i = tid; i < W * nc; i += MG_NT) {
        const int w = i / nc, c = i - w * nc;
        a.seqs[static_cast<int64_t>(r0 + w) * ld + c0 + c] = sm.tile[(sm.nb_row[w] - r0) * TW + c];
        if (sm.f_src[w] >= 0)
          a.fin_tok[static_cast<int64_t>(r0 + w) * ld + c0 + c] = sm.tile[(sm.f_src[w] - r0) * TW + c];
      }
    }
    if (tid < W) a.seqs[static_cast<int64_t>(r0 + tid) * ld + t] = sm.nb_tok[tid];
  }
  // the last sentence of the step reports whether all are finished
  if (tid == 0 && (old_cnt >> 16) == static_cast<unsigned>(a.B - 1)) {
    const int all = static_cast<int>((old_cnt & 0xffffu) + sm.done_now) == a.B;
    *a.all_done_dev = all;
    if (a.all_done_out) *a.all_done_out = all;
    *a.done_count = 0;
  }
}

// ---------------------------------------------------------------------------------------
// reset and finalisation
// ---------------------------------------------------------------------------------------

__global__ void bs_reset_kernel(const BsArgs a) {
  const int64_t n = static_cast<int64_t>(a.R) * a.seq_ld;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % a.seq_ld);
    a.seqs[i] = c == 0 ? a.bos : a.pad;
    a.fin_tok[i] = a.pad;
    if (c == 0) {
      const int r = static_cast<int>(i / a.seq_ld);
      a.scores[r] = (r % a.W) == 0 ? 0.f : -INFINITY;
      a.fin_ns[r] = 0.0;
      a.fin_len[r] = 0;
      a.fin_serial[r] = 0;
      if (r < a.B) {
        a.done[r] = 0;
        a.fin_count[r] = 0;
        a.fin_next[r] = 0;
        a.fin_worst[r] = 1e9;
      }
      if (r == 0) { *a.done_count = 0; *a.all_done_dev = 0; }
    }
  }
}

// One CTA per sentence: add the live beams of unfinished sentences (|y| = steps
// run, normalised by lp_t = lp(steps run)), pick the best normalised score
// (ties: the latest list entry), write the row.
__global__ void bs_finalize_kernel(const BsArgs a, const float* scores, const int32_t* seqs,
                                   int32_t* out_seqs, int32_t* out_len, float* out_score) {
  __shared__ double f_ns[WMAX];
  __shared__ int f_serial[WMAX], f_src[WMAX], f_ntok[WMAX];
  __shared__ int s_best;
  const int b = blockIdx.x;
  const int W = a.W, r0 = b * W, T = a.t, ld = a.seq_ld;
  if (threadIdx.x == 0) {
    int count = a.fin_count[b], next = a.fin_next[b];
    double worst = a.fin_worst[b];
    for (int q = 0; q < W; ++q) {
      f_ns[q] = a.fin_ns[r0 + q];
      f_serial[q] = a.fin_serial[r0 + q];
      f_src[q] = -1;                       // -1: the stored hypothesis in slot q
      f_ntok[q] = a.fin_len[r0 + q];       // an EOS hit at step t holds BOS + t-1 tokens
    }
    if (!a.done[b]) {
      for (int w = 0; w < W; ++w) {
        const double ns = static_cast<double>(scores[r0 + w]) / a.lp_t;
        int slot = -1;
        if (count < W) {
          slot = count++;
          worst = fmin(ns, worst);
        } else if (ns > worst) {
          slot = 0;
          for (int q = 1; q < W; ++q)
            if (f_ns[q] < f_ns[slot] || (f_ns[q] == f_ns[slot] && f_serial[q] < f_serial[slot])) slot = q;
        }
        if (slot >= 0) {
          f_ns[slot] = ns;
          f_serial[slot] = next++;
          f_src[slot] = r0 + w;
          f_ntok[slot] = T + 1;
          if (count >= W) {
            double mn = f_ns[0];
            for (int q = 1; q < W; ++q) mn = fmin(mn, f_ns[q]);
            worst = mn;
          }
        }
      }
    }
    int best = 0;
    for (int q = 1; q < count; ++q)
      if (f_ns[q] > f_ns[best] || (f_ns[q] == f_ns[best] && f_serial[q] > f_serial[best])) best = q;
    s_best = best;
    out_score[b] = static_cast<float>(f_ns[best]);
    const int n = f_ntok[best];
    out_len[b] = (n < ld && a.eos >= 0) ? n + 1 : n;
  }
  __syncthreads();
  const int q = s_best;
  const int n = f_ntok[q];
  const int32_t* src = f_src[q] >= 0 ? seqs + static_cast<int64_t>(f_src[q]) * ld
                                     : a.fin_tok + static_cast<int64_t>(r0 + q) * ld;
  for (int c = threadIdx.x; c < ld; c += blockDim.x) {
    int v = a.pad;
    if (c < n) v = src[c];
    else if (c == n && a.eos >= 0) v = a.eos;
    out_seqs[static_cast<int64_t>(b) * ld + c] = v;
  }
}

// ---------------------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------------------

template <typename T, bool TMA>
static int launch_stream(const BsArgs& a, int grid, cudaStream_t s) {
  static bool attr_set = false;
  const int smem = static_cast<int>(sizeof(BsShared));
  if (!attr_set) {
    if (cudaFuncSetAttribute(bs_stream_kernel<T, TMA>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return VBS_ECUDA;
    attr_set = true;
  }
  bs_stream_kernel<T, TMA><<<grid, BS_NT, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

// The merge grid is a programmatic dependent of the stream grid: it may launch
// while the stream CTAs retire and waits for their writes in griddepcontrol.wait.
static int launch_merge(const BsArgs& a, cudaStream_t s) {
  static bool attr_set = false;
  const int smem = static_cast<int>(sizeof(MergeShared));
  if (!attr_set) {
    if (cudaFuncSetAttribute(bs_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return VBS_ECUDA;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B);
  cfg.blockDim = dim3(MG_NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bs_merge_kernel, a) == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

int launch_bs_step(const BsArgs& a, int grid, bool vector_ok, cudaStream_t s) {
  int st;
  if (a.dtype == VBS_BF16)
    st = vector_ok ? launch_stream<bf16_t, true>(a, grid, s) : launch_stream<bf16_t, false>(a, grid, s);
  else
    st = vector_ok ? launch_stream<float, true>(a, grid, s) : launch_stream<float, false>(a, grid, s);
  if (st != VBS_OK) return st;
  return launch_merge(a, s);
}

int launch_bs_reset(const BsArgs& a, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(a.R) * a.seq_ld;
  const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096));
  bs_reset_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

int launch_bs_finalize(const BsArgs& a, const float* scores, const int32_t* seqs, int32_t* out_seqs,
                       int32_t* out_len, float* out_score, cudaStream_t s) {
  bs_finalize_kernel<<<a.B, 128, 0, s>>>(a, scores, seqs, out_seqs, out_len, out_score);
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

int bs_threads_per_cta() { return BS_NT; }
int bs_ctas_per_sm() { return 1; }

// ---------------------------------------------------------------------------------------
// one expansion step without allocation: its scratch is a static device array
// ---------------------------------------------------------------------------------------

// The partials, row maps and done flags of bs_expand_static.  Every process that loads
// the library holds this array on each device it touches, until it exits.
static __device__ __align__(256) unsigned char g_static_scratch[STATIC_SCRATCH_BYTES];

__global__ void bs_static_prep_kernel(const BsArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < a.R) {
    const int64_t e0 = static_cast<int64_t>(i) * a.V;
    const int64_t p0 = e0 / a.per;
    a.row_p0[i] = static_cast<int>(p0);
    a.row_np[i] = static_cast<int>((e0 + a.V - 1) / a.per - p0 + 1);
  }
  if (i < a.B) a.done[i] = 0;
}

// One CTA per sentence: the rows' partials merged as in bs_merge_kernel, then the W best
// of the sentence's candidates by (score desc, flat index asc) become the new beams.
__global__ void __launch_bounds__(MG_NT) bs_expand_merge_kernel(const BsArgs a, float* scores_out) {
  extern __shared__ __align__(16) unsigned char mg_smem[];
  MergeShared& sm = *reinterpret_cast<MergeShared*>(mg_smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int W = a.W, K = a.K;
  const int r0 = blockIdx.x * W;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int w = warp; w < W; w += MG_NW) row_merge(a, sm, r0 + w, w, lane);
  if (tid < W) { sm.sel_w[tid] = 0; sm.sel_i[tid] = 0; sm.sel_c[tid] = -INFINITY; }
  __syncthreads();
  for (int f = tid; f < W * K; f += MG_NT) {
    const int w = f / K, i = f - w * K;
    if (i >= sm.nval[w]) continue;
    const float c = sm.candv[f];
    int rank = i;
    for (int w2 = 0; w2 < W && rank < W; ++w2)
      if (w2 != w) rank += count_better(sm.candv + w2 * K, sm.nval[w2], c, w2 < w);
    if (rank < W) {
      sm.sel_w[rank] = w;
      sm.sel_i[rank] = i;
      sm.sel_c[rank] = c;
    }
  }
  __syncthreads();
  if (tid < W) {
    const int w = sm.sel_w[tid];
    a.beam_idx[r0 + tid] = r0 + w;
    a.tokens[r0 + tid] = static_cast<int32_t>(key_v(sm.wtop[w * K + sm.sel_i[tid]]));
    scores_out[r0 + tid] = sm.sel_c[tid];
  }
}

namespace {
constexpr int MAX_DEVICES = 256;
std::mutex g_static_mu;
void* g_static_addr[MAX_DEVICES];   // the array's device address, per device ordinal
}  // namespace

int launch_bs_expand_static(BsArgs a, int grid, bool vector_ok, float* scores_out, cudaStream_t s) {
  // carve the array: offsets first, so that an oversized problem is refused before any CUDA call
  size_t off = 0;
  auto take = [&off](size_t bytes) {
    off = (off + 255) & ~static_cast<size_t>(255);
    const size_t at = off;
    off += bytes;
    return at;
  };
  const size_t RP = static_cast<size_t>(a.R) * a.P;
  const size_t o_M = take(RP * sizeof(float));
  const size_t o_l = take(RP * sizeof(float));
  const size_t o_key = take(RP * a.K * sizeof(u64));
  const size_t o_p0 = take(static_cast<size_t>(a.R) * sizeof(int));
  const size_t o_np = take(static_cast<size_t>(a.R) * sizeof(int));
  const size_t o_done = take(static_cast<size_t>(a.B) * sizeof(int));
  if (off > STATIC_SCRATCH_BYTES) return VBS_ESCRATCH;

  // set-up, once per device, with that device current: the array's device address
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return VBS_ECUDA;
  char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return VBS_ECUDA;
      g_static_addr[dev] = p;
    }
    base = static_cast<char*>(g_static_addr[dev]);
  }
  a.part_M = reinterpret_cast<float*>(base + o_M);
  a.part_l = reinterpret_cast<float*>(base + o_l);
  a.part_key = reinterpret_cast<u64*>(base + o_key);
  a.row_p0 = reinterpret_cast<int*>(base + o_p0);
  a.row_np = reinterpret_cast<int*>(base + o_np);
  a.done = reinterpret_cast<int*>(base + o_done);

  const int n = a.R > a.B ? a.R : a.B;
  bs_static_prep_kernel<<<(n + 255) / 256, 256, 0, s>>>(a);
  if (cudaGetLastError() != cudaSuccess) return VBS_ECUDA;
  int st;
  if (a.dtype == VBS_BF16)
    st = vector_ok ? launch_stream<bf16_t, true>(a, grid, s) : launch_stream<bf16_t, false>(a, grid, s);
  else
    st = vector_ok ? launch_stream<float, true>(a, grid, s) : launch_stream<float, false>(a, grid, s);
  if (st != VBS_OK) return st;

  static bool attr_set = false;
  const int smem = static_cast<int>(sizeof(MergeShared));
  if (!attr_set) {
    if (cudaFuncSetAttribute(bs_expand_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return VBS_ECUDA;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B);
  cfg.blockDim = dim3(MG_NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bs_expand_merge_kernel, a, scores_out) == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

}  // namespace vbs
