// Fused batched beam-search step (sm_103a).
//
// The streaming part, shared by both launch shapes: a producer warp streams logit rows
// through a 6-stage ring of 32 KiB shared-memory chunks with bulk (TMA) copies completing
// on mbarriers, and 16 consumer warps read each chunk once: per 32-element tile a thread
// updates an online log-sum-exp (log2 domain, SFU exp2) and compares the tile maximum with
// its row's threshold.  The threshold only takes values that bound the row's K-th best
// logit from below: at a row's first chunk the consumer warps each seed it with the K-th
// best of their lane maxima and meet at a named barrier; a tile whose maximum reaches it
// queues one entry (maximum, column, and a bound on its second-largest value with the
// maximum's place), and one warp per chunk raises it from the queue.  At the end of the
// row the K-th best queued maximum is the final bar; a tile at the bar gives its key from
// its queue entry when its runner-up bound is below the bar, otherwise it is read again.
// A queue overflow falls back to rescanning the row.
//
// bs_cluster_kernel (one launch per step): one thread-block cluster per sentence, each CTA
// streaming whole rows; the sentence's rows meet in distributed shared memory and one warp
// merges them: row LSEs, the best 2W candidates by (score desc, flat index asc), the walk
// that moves EOS hits into the finished set, the stopping test, the outputs and the
// in-place sequence gather.  An instance with FUSE also runs the sentence's paged KV remap.
//
// bs_stream_kernel + bs_merge_kernel (shapes the cluster does not fit): one CTA per SM over
// equal ranges of the flattened [R, V] space, each row segment ending in a partial (max,
// scaled sum, K sorted keys), then one merge CTA per sentence, launched as a programmatic
// dependent.  The same merge finishes the two-pass ablation and the vocabulary-shard path.
//
// No CTA waits on another CTA outside its cluster; every mbarrier wait is bounded.
//
// What is computed follows "Transformers中的Beam Search高效实现" (section
// 多个样本同时进行beam search: log_softmax, add beam_scores, view [batch, W*V],
// top-k, beam_id = j // V, token_id = j % V, BeamHypotheses.add / is_done, pad
// rows of finished sentences) and "9.2 贪心搜索与束搜索" (§9.2.2 four sub-steps,
// "何时结束" early_stopping modes; §9.2.3 length penalty).

#include <cfloat>
#include <cmath>
#include <mutex>

#include <cooperative_groups.h>

#include "common.cuh"
#include "bs_internal.h"
#include "kv_remap.cuh"

namespace vbs {

constexpr int BS_NC = 512;                        // consumer threads
constexpr int BS_NCW = BS_NC / 32;                // consumer warps
constexpr int BS_NT = BS_NC + 32;                 // + the producer warp
constexpr int BS_U = 4;                           // 16-byte vectors per consumer per chunk
constexpr int STAGE_BYTES = BS_NC * BS_U * 16;    // 32 KiB
constexpr int NSTAGE = 6;
constexpr int NSLOT = BS_NSLOT;                   // row segments held before they are published
constexpr int QSEG = 512;                         // candidate queue of one segment
constexpr int QSTEP = 8;                          // threshold refresh once QSTEP more keys are queued
constexpr int FIN_CAP = 64;                       // keys collected at a segment's final bar
constexpr int PF_TILE = 1024;                     // cluster mode: sequence columns prefetched (ints)
constexpr int CT_CAP = 64;                        // tiles re-read at a segment's final bar
constexpr int SEQ_TILE_INTS = 2048;               // sequence gather tile (all W rows)
constexpr int BAR_CONSUMERS = 1;                  // named barrier of the consumer warps
constexpr int MG_NT = 256;                        // merge kernel threads
constexpr int MG_NW = MG_NT / 32;
// fp32 ln 2 split in two: LN2_HI = fl(ln 2), LN2_LO = ln 2 - LN2_HI.
constexpr float LN2_HI = 0.693147182464599609375f;
constexpr float LN2_LO = -1.904654299957768e-09f;

// Two fp32 lanes at once (PTX fma.rn.f32x2 / add.rn.f32x2, sm_100 and later): a0, a1 <-
// a0 * b + c, a1 * b + c; a0, a1 <- a0 + b0, a1 + b1.  Each lane rounds as the scalar op.
__device__ __forceinline__ void fma2(float& a0, float& a1, float b, float c) {
  asm("{.reg .b64 x, y, z; mov.b64 x, {%0, %1}; mov.b64 y, {%2, %2}; mov.b64 z, {%3, %3};"
      " fma.rn.f32x2 x, x, y, z; mov.b64 {%0, %1}, x;}"
      : "+f"(a0), "+f"(a1) : "f"(b), "f"(c));
}
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{.reg .b64 x, y; mov.b64 x, {%0, %1}; mov.b64 y, {%2, %3}; add.rn.f32x2 x, x, y; mov.b64 {%0, %1}, x;}"
      : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1));
}

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

// Descending bitonic sort of 32 keys, one per lane.
__device__ __forceinline__ u64 warp_sort32(u64 key, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const u64 o = shfl64_xor(key, stride);
      const bool take_max = ((lane & stride) == 0) == ((lane & size) == 0);   // size 32: all descending
      key = take_max ? (o > key ? o : key) : (o > key ? key : o);
    }
  }
  return key;
}

// Two descending 32-key lists held one key per lane (0 = none) to the descending 32 best of
// their union: lane i's max(a[i], b[31 - i]) are those 32 and form a bitonic sequence, which
// five compare-exchange stages sort.
__device__ __forceinline__ u64 warp_merge_top32(u64 a, u64 b, int lane) {
  const u64 br = shfl64(b, 31 - lane);
  u64 c = a > br ? a : br;
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) {
    const u64 o = shfl64_xor(c, stride);
    c = (lane & stride) == 0 ? (o > c ? o : c) : (o > c ? c : o);
  }
  return c;
}

// The K best (K <= 32) of n <= QSEG distinct keys (0 = none), in order, into out[0, K):
// the K-th best found bit by bit with warp-wide counts, the keys at or above it gathered one
// per lane and sorted.  out may be overwritten before the end (it holds at most K keys).
__device__ __forceinline__ void warp_topk_bisect(const u64* keys, int n, int K, u64* out, int lane) {
  constexpr int PER = QSEG / 32;
  u64 h[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int j = lane + 32 * i;
    h[i] = j < n ? keys[j] : 0ull;
  }
  u64 x = 0;
  for (int b = 63; b >= 0; --b) {
    const u64 c = x | (1ull << b);
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) cnt += h[i] >= c ? 1 : 0;
    if (__reduce_add_sync(FULL, static_cast<unsigned>(cnt)) >= static_cast<unsigned>(K)) x = c;
  }
  int mine = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) mine += (h[i] != 0ull && h[i] >= x) ? 1 : 0;
  int pos = mine;                                  // inclusive prefix over the lanes
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(FULL, pos, d);
    if (lane >= d) pos += o;
  }
  const int total = __shfl_sync(FULL, pos, 31);
  pos -= mine;
  __syncwarp();
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (h[i] != 0ull && h[i] >= x && pos < K) out[pos++] = h[i];
  __syncwarp();
  u64 v = lane < min(total, K) ? out[lane] : 0ull;
  v = warp_sort32(v, lane);
  __syncwarp();
  if (lane < K) out[lane] = v;
  __syncwarp();
}

// One warp: the K best (K <= 32) of cnt <= 64 distinct keys, in order, into out[0, K): each
// half sorted, then the 32 best of both.
__device__ __forceinline__ void warp_sort_top64(const u64* keys, int cnt, int K, u64* out, int lane) {
  const u64 k0 = lane < cnt ? keys[lane] : 0ull;
  const u64 k1 = lane + 32 < cnt ? keys[lane + 32] : 0ull;
  const u64 t = warp_merge_top32(warp_sort32(k0, lane), warp_sort32(k1, lane), lane);
  __syncwarp();
  if (lane < K) out[lane] = t;
}

// K best of nl descending lists of K keys each (keys distinct, 0 = none), in order: K rounds
// of a warp-wide maximum over the lists' heads; lane c walks lists c, c + 32, ...
// (nl <= PART_KEYS / 2).
__device__ void warp_merge_sorted(const u64* lists, int nl, int K, u64* out, int lane) {
  constexpr int LPL = PART_KEYS / 2 / 32;
  int pos[LPL];
  u64 head[LPL];
#pragma unroll
  for (int m = 0; m < LPL; ++m) {
    const int c = lane + 32 * m;
    pos[m] = 0;
    head[m] = c < nl ? lists[c * K] : 0ull;
  }
  for (int i = 0; i < K; ++i) {
    u64 mine = head[0];
#pragma unroll
    for (int m = 1; m < LPL; ++m) mine = head[m] > mine ? head[m] : mine;
    const u32 hi = static_cast<u32>(mine >> 32);
    const u32 mhi = __reduce_max_sync(FULL, hi);
    const u32 mlo = __reduce_max_sync(FULL, hi == mhi ? static_cast<u32>(mine) : 0u);
    const u64 best = (static_cast<u64>(mhi) << 32) | mlo;
    if (lane == 0) out[i] = best;
    if (best != 0ull) {
#pragma unroll
      for (int m = 0; m < LPL; ++m) {
        if (head[m] == best) {                 // the one list it came from moves on
          ++pos[m];
          head[m] = pos[m] < K ? lists[(lane + 32 * m) * K + pos[m]] : 0ull;
        }
      }
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------------------
// shared memory
// ---------------------------------------------------------------------------------------

struct BsShared {                              // the stream kernel
  unsigned char ring[NSTAGE][STAGE_BYTES];     // the streamed chunks
  u64 q[NSLOT][QSEG];                          // hot tiles (max, position) per row segment; keys after a rescan
  u32 qd[NSLOT][QSEG];                         // per hot tile: a bound on its second-largest value | max's place
  u64 fin[NSLOT][FIN_CAP];                     // a segment's final candidate keys
  u32 ctile[NSLOT][CT_CAP];                    // a segment's final candidate tiles (queue indices)
  float M[NSLOT][BS_NCW], l[NSLOT][BS_NCW];    // per-warp (max, scaled sum) of each segment
  u64 full[NSTAGE], empty[NSTAGE];
  u64 rbar[NSLOT];                             // the key bar of a rescan
  u32 thr[NSLOT];                              // threshold (ordered logit bits) per segment
  u32 tmin[NSLOT];                             // first chunk: the least of the warps' ceil(K / warps)-th best
  u32 sbar[NSLOT];                             // the final bar (ordered logit bits)
  int qcnt[NSLOT];                             // entries reserved in q[slot] (> QSEG: overflow)
  int qref[NSLOT];                             // qcnt at the last threshold refresh
  int fcnt[NSLOT];                             // keys found at the final bar
  int mode[NSLOT];                             // 0: tiles resolved, 1: needs a rescan, 2: q holds keys
  int seg_r[NSLOT], seg_v0[NSLOT], seg_v1[NSLOT], seg_skip[NSLOT];
  int stage_skip[NSTAGE];                      // the producer's skip decision for each ring stage
  // cluster mode: this CTA's whole rows (K best keys, sorted; max and scaled sum)
  u64 rk[NSLOT][KMAX];
  float rM[NSLOT], rl[NSLOT];
  // cluster mode: the sentence merge's candidates (one per lane)
  u64 cm_key[32];
  float cm_c[32];
  int cm_w[32], cm_sel[32];
  // cluster mode: the merge's decisions, read by every thread of the first CTA for the gather
  int cm_nbrow[WMAX], cm_fsrc[WMAX], cm_nbtok[WMAX];
  int cm_gather;
  // cluster mode: the merge's inputs this kernel does not write, prefetched at its start
  int pf_tile[PF_TILE];
  double pf_fns[WMAX], pf_fworst;
  float pf_s[WMAX];
  int pf_flen[WMAX], pf_fser[WMAX], pf_fcount, pf_fnext, pf_done;
};

static_assert(sizeof(BsShared) <= 232448, "the stream kernel's shared memory fits one SM");
constexpr int REMAP_SH_BYTES = (static_cast<int>(sizeof(RemapShared)) + 15) / 16 * 16;

// The cluster kernel can run a sentence's paged KV remap after its merge when the remap's
// shared state fits in the (then idle) ring.
bool bs_can_fuse_remap(const BsArgs& a, const PagedArgs& kv) {
  return a.cluster != 0 && kv.B == a.B && kv.W == a.W &&
         REMAP_SH_BYTES + remap_scratch_ints(kv) * 4 <= static_cast<int64_t>(sizeof(BsShared::ring));
}

struct MergeShared {                           // the merge kernel
  u64 rowscratch[WMAX * PART_KEYS];            // the rows' partial lists
  float pM[PART_KEYS / 2], pL[PART_KEYS / 2];  // the rows' partial (max, sum): W * P <= PART_KEYS / 2
  int np[WMAX];                                // partials per row
  u64 wtop[WMAX * KMAX];                       // the W rows' sorted lists
  float candv[WMAX * KMAX];                    // their candidate scores, list order
  int nval[WMAX];
  int sel_w[KMAX], sel_i[KMAX];                // the sentence's best 2W, in order
  float sel_c[KMAX];
  int tile[SEQ_TILE_INTS];                     // the parents' sequence rows
  float s[WMAX];
  float f_ns[WMAX];                            // normalised scores (all float-representable)
  int f_len[WMAX], f_serial[WMAX], f_src[WMAX];
  int f_count, f_next;
  float f_worst;
  float nb_score[WMAX];
  int nb_tok[WMAX], nb_row[WMAX];
  int done_now;
};

// ---------------------------------------------------------------------------------------
// thresholds and the hot-tile queues
// ---------------------------------------------------------------------------------------
//
// A lane whose tile (BS_U vectors of one chunk) has a maximum at or above the segment's
// threshold queues one entry: (ordered bits of the tile maximum, first column of the
// tile).  Tile maxima are logits of distinct elements, so the K-th best queued maximum is
// a lower bound of the segment's K-th best logit; the threshold only ever takes such
// values.  At the end, every element at or above the final bar (the K-th best queued
// maximum) lies in a queued tile whose maximum reaches the bar: only those few tiles are
// read again, from global memory, to find the segment's exact K best keys.

// The rank of each lane's value among the warp's 32 (the lanes before it: a larger
// value, or the same value in a lower lane); the ranks are 0..31, once each.
__device__ __forceinline__ int warp_rank_u32(u32 v, int lane) {
  int rank = 0;
#pragma unroll
  for (int i = 1; i < 32; ++i) {
    const int src = (lane + i) & 31;
    const u32 o = __shfl_sync(FULL, v, src);
    rank += (o > v || (o == v && src < lane)) ? 1 : 0;
  }
  return rank;
}

// The K-th largest of the warp's 32 lane values (repeats counted; K <= 32), 0 if fewer
// than K lanes hold a nonzero value.
__device__ __forceinline__ u32 warp_kth_u32(u32 v, int K, int lane) {
  const u32 b = __ballot_sync(FULL, warp_rank_u32(v, lane) == K - 1);
  return __shfl_sync(FULL, v, __ffs(b) - 1);
}

// warp_kth_u32 out of line, for the K <= 8 streaming loop's once-per-row seed: the hot loop's
// code stays smaller for the instruction caches (measured 3 % faster at the Llama shape; the
// K > 8 instance measured slower with it and keeps the seed inline).
__device__ __noinline__ u32 warp_kth_u32_cold(u32 v, int K, int lane) { return warp_kth_u32(v, K, lane); }

// Warp-wide: the K-th best of the lane maxima of the first n entries' tile maxima (0 if
// fewer than K lanes hold one).  An entry another warp has reserved but not written yet
// reads 0 and is ignored.
template <class SH>
__device__ __forceinline__ u32 queue_bar(const SH& sh, int slot, int n, int K, int lane) {
  const volatile u64* vq = sh.q[slot];
  u32 lm = 0;
  for (int j = lane; j < n; j += 32) {
    const u32 h = static_cast<u32>(vq[j] >> 32);
    lm = h > lm ? h : lm;
  }
  return warp_kth_u32(lm, K, lane);
}

// Warp-wide, for lists longer than a warp's lanes make tight (K > 8): the largest x whose
// low 32 - bits bits are zero with at least K of the first n entries' tile maxima at or
// above it, found bit by bit from the top; with bits = 32 it is their K-th best exactly
// (0 if fewer than K are nonzero).
template <class SH>
__device__ __forceinline__ u32 queue_kth(const SH& sh, int slot, int n, int K, int lane, int bits) {
  constexpr int PER = QSEG / 32;
  const volatile u64* vq = sh.q[slot];
  u32 h[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int j = lane + 32 * i;
    h[i] = j < n ? static_cast<u32>(vq[j] >> 32) : 0u;
  }
  u32 x = 0;
  for (int b = 31; b >= 32 - bits; --b) {
    const u32 c = x | (1u << b);
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) cnt += h[i] >= c ? 1 : 0;
    if (__reduce_add_sync(FULL, static_cast<unsigned>(cnt)) >= static_cast<unsigned>(K)) x = c;
  }
  return x;
}

// Warp-wide: raise the segment's threshold from its queue.
template <bool BIGK, class SH>
__device__ __noinline__ void queue_refresh(SH& sh, int slot, int n, int K, int lane) {
  if (lane == 0) sh.qref[slot] = n;
  const u32 t = BIGK ? queue_kth(sh, slot, n, K, lane, 20) : queue_bar(sh, slot, n, K, lane);
  if (lane == 0 && t) atomicMax(&sh.thr[slot], t);
}

// ---------------------------------------------------------------------------------------
// the stream kernel's parts
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

// Read through L2: other SMs wrote both in the previous step.
__device__ __forceinline__ bool row_skipped(const BsArgs& a, int r) {
  return __ldcg(a.done + r / a.W) != 0 || __ldcg(a.scores + r) == -INFINITY;
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
    u32 bytes = skip ? 0u : static_cast<u32>(ch.len * Elem<T>::BYTES);
    if (bytes && !VBS_CHECK(ch.r < a.R && ch.v0 >= 0 && ch.v0 + ch.len <= a.V, 1, ch.r, a.status)) bytes = 0;
    sh.stage_skip[slot] = skip ? 1 : 0;               // published by the arrive below
    mbar_expect_tx(&sh.full[slot], bytes);
    if (bytes) {
      const char* src = reinterpret_cast<const char*>(a.logits) +
                        (static_cast<int64_t>(ch.r) * a.ld + ch.v0) * Elem<T>::BYTES;
      bulk_g2s(sh.ring[slot], src, bytes, &sh.full[slot]);
    }
  }
}

// One warp: resolve segment s from its queue.  The final bar is the K-th best queued tile
// maximum; the tiles reaching it are read again and every element at or above the bar
// is collected into fin[s].  mode[s] becomes 1 when that does not fit (queue overflow,
// more than CT_CAP tiles or FIN_CAP keys at the bar: ties, adversarial orders).
template <typename T, int VEC, bool BIGK, class SH>
__device__ void resolve_tiles(const BsArgs& a, SH& sh, int s, int lane) {
  const int K = a.K;
  const int qn = sh.qcnt[s];
  const int n = min(qn, QSEG);
  const u32 bar = BIGK ? queue_kth(sh, s, n, K, lane, 32) : queue_bar(sh, s, n, K, lane);
  if (lane == 0) { sh.sbar[s] = bar; sh.fcnt[s] = 0; }
  int nc = 0;
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    const u64 e = j < n ? sh.q[s][j] : 0ull;
    const bool cand = e != 0 && static_cast<u32>(e >> 32) >= bar;
    const u32 b = __ballot_sync(FULL, cand);
    const int pos = nc + __popc(b & ((1u << lane) - 1u));
    if (cand && pos < CT_CAP) sh.ctile[s][pos] = static_cast<u32>(j);
    nc += __popc(b);
  }
  __syncwarp();
  if (qn > QSEG || nc > CT_CAP) {
    if (lane == 0) sh.mode[s] = 1;
    return;
  }
  const float bar_x = bar ? unord_f32(bar) : -INFINITY;
  const int sv1 = sh.seg_v1[s];
  const char* row = reinterpret_cast<const char*>(a.logits) + static_cast<int64_t>(sh.seg_r[s]) * a.ld * Elem<T>::BYTES;
  for (int t = lane; t < nc; t += 32) {
    const int jq = static_cast<int>(sh.ctile[s][t]);
    const u64 eq = sh.q[s][jq];
    const u32 vb = static_cast<u32>(eq);
    const u32 desc = sh.qd[s][jq];
    if ((desc & ~31u) <= bar) {
      // every other element of the tile lies below the bar: the maximum is the only key
      const u32 pu = (desc & 31u) / VEC, pe = (desc & 31u) % VEC;
      const int p = atomicAdd(&sh.fcnt[s], 1);
      if (p < FIN_CAP) sh.fin[s][p] = make_key(unord_f32(static_cast<u32>(eq >> 32)), vb + pu * (BS_NC * VEC) + pe);
      continue;
    }
#pragma unroll
    for (int u = 0; u < BS_U; ++u) {
      const u32 v0 = vb + static_cast<u32>(u * BS_NC * VEC);
      if (v0 >= static_cast<u32>(sv1)) continue;
      float x[VEC];
      if constexpr (VEC == 1) {
        x[0] = Elem<T>::load(row, v0);
      } else {
        Vec16<T>::unpack(ld_stream16(row + static_cast<int64_t>(v0) * Elem<T>::BYTES), x);
      }
#pragma unroll
      for (int e2 = 0; e2 < VEC; ++e2) {
        if (x[e2] >= bar_x) {
          const int p = atomicAdd(&sh.fcnt[s], 1);
          if (p < FIN_CAP) sh.fin[s][p] = make_key(x[e2], v0 + e2);
        }
      }
    }
  }
  __syncwarp();
  if (lane == 0) sh.mode[s] = sh.fcnt[s] > FIN_CAP ? 1 : 0;
}

// All consumers, for a segment resolve_tiles could not finish: collect every key of the
// segment at or above a bar, re-reading the segment from global memory, until one pass
// fits in the queue; each pass that overflows raises the bar to the K-th best key it
// queued (keys are distinct and QSEG > K, so the bar rises and the passes end).  Only
// ties at the bar and adversarial orders (e.g. ascending logits) get here.  The aligned
// path reads 16-byte vectors: the segment may have left L2 by now.
template <typename T, int VEC, bool BIGK>
__device__ void rescan_segment(const BsArgs& a, BsShared& sh, int s) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  const int r = sh.seg_r[s], sv0 = sh.seg_v0[s], sv1 = sh.seg_v1[s];
  const char* row = reinterpret_cast<const char*>(a.logits) + static_cast<int64_t>(r) * a.ld * Elem<T>::BYTES;
  if (tid == 0) sh.rbar[s] = static_cast<u64>(sh.sbar[s]) << 32;
  for (;;) {
    named_sync(BAR_CONSUMERS, BS_NC);
    const u64 bar = sh.rbar[s];
    for (int i = tid; i < QSEG; i += BS_NC) sh.q[s][i] = 0ull;
    if (tid == 0) sh.qcnt[s] = 0;
    named_sync(BAR_CONSUMERS, BS_NC);
    for (int v = sv0 + tid * VEC; v < sv1; v += BS_NC * VEC) {
      float x[VEC];
      if constexpr (VEC == 1) x[0] = Elem<T>::load(row, v);
      else Vec16<T>::unpack(ld_stream16(row + static_cast<int64_t>(v) * Elem<T>::BYTES), x);
#pragma unroll
      for (int e2 = 0; e2 < VEC; ++e2) {
        const u64 k = make_key(x[e2], static_cast<u32>(v + e2));
        if (k >= bar) {
          const int pos = atomicAdd(&sh.qcnt[s], 1);
          if (pos < QSEG) sh.q[s][pos] = k;
        }
      }
    }
    named_sync(BAR_CONSUMERS, BS_NC);
    if (sh.qcnt[s] <= QSEG) break;
    if (warp == 0) {
      if constexpr (BIGK) warp_topk_bisect(sh.q[s], QSEG, K, sh.fin[s], lane);
      else warp_select_topk(sh.q[s], QSEG, K, sh.fin[s], lane);
      if (lane == 0) sh.rbar[s] = sh.fin[s][K - 1];
    }
  }
  if (tid == 0) sh.mode[s] = 2;
  named_sync(BAR_CONSUMERS, BS_NC);
}

// One warp: segment s's partial -- (max, scaled sum) over the warps and its K best keys,
// sorted -- written to its slot of the row's partials; then the slot is cleared.
template <bool BIGK>
__device__ void finish_segment(const BsArgs& a, BsShared& sh, int s, int lane) {
  const int K = a.K;
  const int mode = sh.mode[s];
  if (!sh.seg_skip[s]) {
    float Mw = lane < BS_NCW ? sh.M[s][lane] : -INFINITY;
    float lw = lane < BS_NCW ? sh.l[s][lane] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float M2 = __shfl_xor_sync(FULL, Mw, off);
      const float l2 = __shfl_xor_sync(FULL, lw, off);
      lse_merge(Mw, lw, M2, l2);
    }
    const int r = sh.seg_r[s];
    const int64_t pslot =
        a.cluster ? 0 : static_cast<int64_t>(r) * a.P + (static_cast<int>(blockIdx.x) - a.row_p0[r]);
    const bool pslot_ok = VBS_CHECK(pslot >= 0 && pslot < static_cast<int64_t>(a.R) * a.P, 2, pslot, a.status);
    u64* out = a.cluster ? sh.rk[s] : (pslot_ok ? a.part_key + pslot * K : sh.fin[s]);   // cluster mode: in shared memory
    if (mode == 0) {
      const int cnt = sh.fcnt[s];
      if (!BIGK || cnt <= 16) {
        for (int j = lane; j < cnt; j += 32) {
          const u64 k = sh.fin[s][j];
          int rank = 0;
          for (int i = 0; i < cnt; ++i) rank += sh.fin[s][i] > k;
          if (rank < K) out[rank] = k;
        }
        if (lane < K && lane >= cnt) out[lane] = 0ull;
      } else if constexpr (BIGK) {
        warp_sort_top64(sh.fin[s], cnt, K, out, lane);   // up to FIN_CAP = 64 keys
      }
    } else {
      if constexpr (BIGK) warp_topk_bisect(sh.q[s], min(sh.qcnt[s], QSEG), K, sh.fin[s], lane);
      else warp_select_topk(sh.q[s], min(sh.qcnt[s], QSEG), K, sh.fin[s], lane);
      if (lane < K) out[lane] = sh.fin[s][lane];
    }
    if (lane == 0) {
      if (a.cluster) {
        sh.rM[s] = Mw;
        sh.rl[s] = lw;
      } else if (pslot_ok) {
        a.part_M[pslot] = Mw;
        a.part_l[pslot] = lw;
      }
    }
  }
  __syncwarp();
  const int n = mode == 0 ? min(sh.qcnt[s], QSEG) : QSEG;
  for (int j = lane; j < n; j += 32) sh.q[s][j] = 0ull;
  if (lane == 0) { sh.qcnt[s] = 0; sh.qref[s] = 0; sh.thr[s] = 0u; sh.tmin[s] = 0xffffffffu; sh.mode[s] = 0; }
}

// All consumers (after a consumer barrier): publish slots [0, ns).
// Warp s resolves slot s and, unless its queue must be rescanned, finishes it at once; the
// rescans (every consumer thread) follow the one barrier, each finished by its slot's warp.
template <typename T, int VEC, bool BIGK>
__device__ void publish_slots(const BsArgs& a, BsShared& sh, int ns) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp < ns) {
    if (!sh.seg_skip[warp]) resolve_tiles<T, VEC, BIGK>(a, sh, warp, lane);
    __syncwarp();
    if (sh.seg_skip[warp] || sh.mode[warp] != 1) finish_segment<BIGK>(a, sh, warp, lane);
  }
  named_sync(BAR_CONSUMERS, BS_NC);
  for (int s = 0; s < ns; ++s) {
    if (!sh.seg_skip[s] && sh.mode[s] == 1) {      // the same for every thread
      rescan_segment<T, VEC, BIGK>(a, sh, s);
      if (warp == s) finish_segment<BIGK>(a, sh, s, lane);
    }
  }
}

// publish_slots out of line, for the K <= 8 streaming loop's publish when every slot holds a
// segment (the stream kernel's long ranges): inlined, its resolve, finish and rescan code
// enlarged the loop's code (3 % slower at the Llama shape, where it never runs).
template <typename T, int VEC, bool BIGK>
__device__ __noinline__ void publish_slots_cold(const BsArgs& a, BsShared& sh, int ns) {
  publish_slots<T, VEC, BIGK>(a, sh, ns);
}

// The consumers: every chunk of the range, one row segment after the other.  Nothing in
// the loop waits for another warp; segments are published after the loop (or when all
// NSLOT slots hold one).
// BIGK (the stream kernel's instance for K > 8): the threshold seed takes a second,
// cross-warp bound and the queue's bars are computed exactly.
template <typename T, bool TMA, bool BIGK>
__device__ void consume(const BsArgs& a, BsShared& sh, int64_t e0, int64_t e1) {
  constexpr int VEC = TMA ? Vec16<T>::N : 1;
  constexpr int64_t SE = static_cast<int64_t>(BS_NC) * BS_U * VEC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  float M = -INFINITY, m = -INFINITY, l = 0.f;
  bool skip = false, seeded = false;
  int seg = -1, slot = 0;
  int rs = 0;                                       // ring stage of chunk c, and its phase
  u32 ph = 0;
  ChunkCursor cur(e0, e1, a.V, static_cast<int>(SE));
  for (int c = 0; cur.more(); ++c) {
    const Chunk ch = cur.next();
    if (ch.first) {
      ++seg;
      slot = seg % NSLOT;
      if (seg > 0 && slot == 0) {                   // every slot holds a segment: publish them
        named_sync(BAR_CONSUMERS, BS_NC);
        if constexpr (BIGK) publish_slots<T, VEC, BIGK>(a, sh, NSLOT);   // K > 8: frequent, kept inline
        else publish_slots_cold<T, VEC, BIGK>(a, sh, NSLOT);
        named_sync(BAR_CONSUMERS, BS_NC);
      }
      if constexpr (!TMA) skip = row_skipped(a, ch.r);
      M = -INFINITY;
      m = -INFINITY;
      l = 0.f;
      seeded = false;
    }
    const int n = ch.len / VEC;                     // vectors in this chunk
    uint4 q[BS_U];
    float xs[BS_U];
    if constexpr (TMA) {
      if (!mbar_wait(&sh.full[rs], ph)) set_status(a.status, VBS_ETIMEOUT);
      skip = sh.stage_skip[rs] != 0;                // the producer's decision for this row
      const uint4* stage = reinterpret_cast<const uint4*>(sh.ring[rs]) + tid;
      if (!skip && n == BS_NC * BS_U) {             // a full chunk: no per-vector bounds
#pragma unroll
        for (int u = 0; u < BS_U; ++u) q[u] = stage[u * BS_NC];
      } else {
#pragma unroll
        for (int u = 0; u < BS_U; ++u) {
          const int i = tid + u * BS_NC;
          constexpr u32 NEG = VecMax<T>::NEG;
          q[u] = (!skip && i < n) ? stage[u * BS_NC] : make_uint4(NEG, NEG, NEG, NEG);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[rs]);    // the stage may refill once every warp has its data
      if (++rs == NSTAGE) { rs = 0; ph ^= 1u; }
    } else {
      const char* row = reinterpret_cast<const char*>(a.logits) +
                        (static_cast<int64_t>(ch.r) * a.ld + ch.v0) * Elem<T>::BYTES;
#pragma unroll
      for (int u = 0; u < BS_U; ++u) {
        const int i = tid + u * BS_NC;
        xs[u] = (!skip && i < n) ? Elem<T>::load(row, i) : -INFINITY;
      }
    }
    if (ch.first && tid == 0) {
      sh.seg_r[slot] = ch.r;
      sh.seg_v0[slot] = ch.v0;
      sh.seg_skip[slot] = skip ? 1 : 0;
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
      // the threshold: each warp seeds it at the segment's first chunk with the K-th best
      // of its lane maxima; one warp per chunk raises it from the queue once QSTEP more
      // tiles have been queued
      u32 thr_o = *reinterpret_cast<volatile u32*>(&sh.thr[slot]);
      const u32 tmo = tm > -INFINITY ? ord_f32(tm) : 0u;
      if (!seeded) {
        // every consumer warp is at the segment's first chunk: the threshold starts at
        // the best of the warps' seeds, so only a few tiles of this chunk are queued
        seeded = true;
        const u32 seed = BIGK ? warp_kth_u32(tmo, K, lane) : warp_kth_u32_cold(tmo, K, lane);
        if (lane == 0 && seed > thr_o) atomicMax(&sh.thr[slot], seed);
        if constexpr (BIGK) {
          // a second bound: each of the BS_NCW warps has j = ceil(K / BS_NCW) lane maxima
          // at or above its own j-th best, so at least K tiles reach the least of those
          // (with K > 8 the warps' K-th bests alone let most of the chunk's tiles in)
          const u32 seed_j = warp_kth_u32(tmo, (K + BS_NCW - 1) / BS_NCW, lane);
          if (lane == 0) atomicMin(&sh.tmin[slot], seed_j);
        }
        named_sync(BAR_CONSUMERS, BS_NC);
        thr_o = *reinterpret_cast<volatile u32*>(&sh.thr[slot]);
        if constexpr (BIGK) {
          const u32 mn = *reinterpret_cast<volatile u32*>(&sh.tmin[slot]);
          if (mn > thr_o) {
            thr_o = mn;
            if (lane == 0) atomicMax(&sh.thr[slot], mn);
          }
        }
      }
      if (tmo != 0u && tmo >= thr_o) {
        // also record where the maximum sits (vector um, element em) and a bound on the
        // tile's second-largest value, so that the final resolve seldom reads the tile
        // again; signed zeros compare equal as floats, so a zero maximum or runner-up
        // leaves the descriptor unknown
        int um = -1, em = -1;
        float sec = -INFINITY;
        uint4 qm = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < BS_U; ++u) {
          float vmu;
          if constexpr (TMA) vmu = VecMax<T>::finish(VecMax<T>::fold(q[u], VecMax<T>::NEG));
          else vmu = xs[u];
          const bool hit = um < 0 && vmu == tm;
          if (hit) {
            um = u;
            if constexpr (TMA) qm = q[u];
            else qm.x = __float_as_uint(xs[u]);
          } else {
            sec = fmaxf(sec, vmu);
          }
        }
        float x[VEC];
        if constexpr (TMA) Vec16<T>::unpack(qm, x);
        else x[0] = __uint_as_float(qm.x);
#pragma unroll
        for (int e2 = 0; e2 < VEC; ++e2) {
          const bool hit = em < 0 && x[e2] == tm;
          if (hit) em = e2;
          else sec = fmaxf(sec, x[e2]);
        }
        const u32 so = sec > -INFINITY ? ord_f32(sec) : 0u;
        const bool known = um >= 0 && em >= 0 && tm != 0.0f && sec != 0.0f && so < 0xffffffe0u;
        const u32 desc = known ? (((so >> 5) + 1u) << 5) | static_cast<u32>(um * VEC + em) : 0xffffffffu;
        const int pos = atomicAdd(&sh.qcnt[slot], 1);
        if (pos < QSEG) {
          sh.q[slot][pos] = (static_cast<u64>(tmo) << 32) | static_cast<u32>(ch.v0 + tid * VEC);
          sh.qd[slot][pos] = desc;
        }
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
          if constexpr (VEC == 8) {                // bf16: the exponents' arguments and sums in pairs
#pragma unroll
            for (int e2 = 0; e2 < VEC; e2 += 2) fma2(x[e2], x[e2 + 1], LOG2E_F, -M);
#pragma unroll
            for (int e2 = 0; e2 < VEC; ++e2) x[e2] = ex2(x[e2]);
            add2(x[0], x[1], x[2], x[3]);
            add2(x[4], x[5], x[6], x[7]);
            add2(x[0], x[1], x[4], x[5]);
            acc[u] = x[0] + x[1];
          } else {
#pragma unroll
            for (int e2 = 0; e2 < VEC; ++e2) x[e2] = ex2(fmaf(x[e2], LOG2E_F, -M));
#pragma unroll
            for (int w = 1; w < VEC; w <<= 1)
#pragma unroll
              for (int e2 = 0; e2 + w < VEC; e2 += 2 * w) x[e2] += x[e2 + w];
            acc[u] = x[0];
          }
        }
#pragma unroll
        for (int w = 1; w < BS_U; w <<= 1)
#pragma unroll
          for (int u = 0; u + w < BS_U; u += 2 * w) acc[u] += acc[u + w];
        l += acc[0];
      }
      if (warp == (c & (BS_NCW - 1))) {
        const int nq = __shfl_sync(FULL, *reinterpret_cast<volatile int*>(&sh.qcnt[slot]), 0);
        const int nr = __shfl_sync(FULL, *reinterpret_cast<volatile int*>(&sh.qref[slot]), 0);
        if (nq >= nr + QSTEP) queue_refresh<BIGK>(sh, slot, nq < QSEG ? nq : QSEG, K, lane);
      }
    }
    if (ch.last) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float M2 = __shfl_xor_sync(FULL, M, off);
        const float l2 = __shfl_xor_sync(FULL, l, off);
        lse_merge(M, l, M2, l2);
      }
      if (lane == 0) { sh.M[slot][warp] = M; sh.l[slot][warp] = l; }
      if (tid == 0) sh.seg_v1[slot] = ch.v0 + ch.len;
    }
  }
  named_sync(BAR_CONSUMERS, BS_NC);
  if (seg >= 0) publish_slots<T, VEC, BIGK>(a, sh, slot + 1);
}

// ---------------------------------------------------------------------------------------
// the stream kernel
// ---------------------------------------------------------------------------------------

template <typename T, bool TMA, bool BIGK>
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
    if (threadIdx.x < NSLOT) {
      sh.thr[threadIdx.x] = 0u;
      sh.tmin[threadIdx.x] = 0xffffffffu;
      sh.qcnt[threadIdx.x] = 0;
      sh.qref[threadIdx.x] = 0;
      sh.mode[threadIdx.x] = 0;
    }
    for (int i = threadIdx.x; i < NSLOT * QSEG; i += BS_NT) (&sh.q[0][0])[i] = 0ull;
    __syncthreads();
    if ((threadIdx.x >> 5) == BS_NCW) {
      if constexpr (TMA) {
        if ((threadIdx.x & 31) == 0) produce<T>(a, sh, e0, e1);
      }
    } else {
      consume<T, TMA, BIGK>(a, sh, e0, e1);
    }
  }
  // the merge grid may start filling the SMs this CTA leaves
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}


// ---------------------------------------------------------------------------------------
// cluster mode: a cluster of C CTAs per sentence, each CTA streaming W/C whole rows
// ---------------------------------------------------------------------------------------
//
// When W * 2W <= 32 and B * C CTAs fit one wave, sentence b is owned by the cluster of C
// CTAs b*C .. b*C+C-1, CTA c streaming rows b*W + c*(W/C) .. + W/C - 1 whole.  Each CTA
// leaves its rows' K best keys and (max, scaled sum) in its own shared memory; after a
// cluster barrier one warp of the cluster's first CTA reads them through distributed
// shared memory and merges the sentence: no partials in global memory, no second kernel.

constexpr int CM_TILE = 8192;                      // sequence staging (ints), in the free ring

__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" :: "r"(smem_u32(smem)), "l"(gmem) : "memory");
}

// One warp of the cluster's first CTA, at the kernel's start: the sentence state and the
// first sequence columns (written by earlier kernels only) are copied into shared memory
// asynchronously, to be ready when the merge needs them.
__device__ void cluster_prefetch(const BsArgs& a, BsShared& sh, int b, int lane) {
  const int W = a.W, r0 = b * W, ld = a.seq_ld;
  const int TWp = PF_TILE / W;
  const int nc = min(a.t, TWp);
  for (int i = lane; i < W * nc; i += 32) {
    const int w = i / nc, c = i - w * nc;
    cp_async4(&sh.pf_tile[w * TWp + c], a.seqs + static_cast<int64_t>(r0 + w) * ld + c);
  }
  if (lane < W) {
    cp_async4(&sh.pf_s[lane], a.scores + r0 + lane);
    cp_async8(&sh.pf_fns[lane], a.fin_ns + r0 + lane);
    cp_async4(&sh.pf_flen[lane], a.fin_len + r0 + lane);
    cp_async4(&sh.pf_fser[lane], a.fin_serial + r0 + lane);
  }
  if (lane == 0) {
    cp_async4(&sh.pf_fcount, a.fin_count + b);
    cp_async4(&sh.pf_fnext, a.fin_next + b);
    cp_async8(&sh.pf_fworst, a.fin_worst + b);
    cp_async4(&sh.pf_done, a.done + b);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// One warp: sentence b's merge from the cluster's row results (W * K <= 32; lane = w*K + i).
// Lane 0 returns the step's finished-sentence count before this sentence (old_cnt) and
// whether it is done now; the sequence gather is left to cluster_gather.
__device__ void cluster_merge_sentence(const BsArgs& a, BsShared& sh, int b, int lane, unsigned& old_cnt,
                                       int& done_now) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int W = a.W, K = a.K, RPC = W / a.cluster;
  const int r0 = b * W, t = a.t, ld = a.seq_ld;
  // ---- one round of loads: the rows' results (distributed shared memory), the sentence state
  const int wl = min(lane / K, W - 1), il = lane - wl * K;
  u64 kl = 0ull;
  if (lane < W * K) kl = cl.map_shared_rank(&sh, wl / RPC)->rk[wl % RPC][il];
  asm volatile("cp.async.wait_all;" ::: "memory");   // this warp's prefetch of the sentence state
  __syncwarp();
  float Mr = -INFINITY, lr = 0.f, s_row = 0.f, fns = 0.f;
  int flen = 0, fser = 0;
  if (lane < W) {
    const BsShared* src = cl.map_shared_rank(&sh, lane / RPC);
    Mr = src->rM[lane % RPC];
    lr = src->rl[lane % RPC];
    s_row = sh.pf_s[lane];
    fns = static_cast<float>(sh.pf_fns[lane]);
    flen = sh.pf_flen[lane];
    fser = sh.pf_fser[lane];
  }
  int fcount = sh.pf_fcount, fnext = sh.pf_fnext;
  float fworst = static_cast<float>(sh.pf_fworst);
  const bool was_done = sh.pf_done != 0;
  old_cnt = 0;
  done_now = 1;
  int nb_row = r0, nb_tok = a.pad, f_src = -1;     // lane w < W: new beam w, finished slot w's source
  float nb_score = 0.f;
  if (!was_done) {
    // ---- row LSEs as fp32 pairs hi + lo (lanes < W), then the candidates' scores
    float hi = 0.f, lo = 0.f;
    if (lane < W && s_row != -INFINITY) {
      const float L2 = log2f(lr);
      const float t_hi = Mr + L2;
      const float bb = t_hi - Mr;
      const float t_lo = (Mr - (t_hi - bb)) + (L2 - bb);
      const float p2 = t_hi * LN2_HI;
      const float e = fmaf(t_hi, LN2_HI, -p2) + fmaf(t_hi, LN2_LO, t_lo * LN2_HI);
      hi = p2 + e;
      lo = e - (hi - p2);
      if (!(hi > -INFINITY && hi < INFINITY)) set_status(a.status, VBS_EINPUT);  // no finite logit, NaN, +inf
    }
    const float sw = __shfl_sync(FULL, s_row, wl);
    const float hw = __shfl_sync(FULL, hi, wl), lw = __shfl_sync(FULL, lo, wl);
    float cl_ = -INFINITY;
    if (lane < W * K) {
      if (sw == -INFINITY) {                       // a row at -inf: -inf candidates by token id
        kl = il < min(K, a.V) ? make_key(-INFINITY, static_cast<u32>(il)) : 0ull;
      } else {
        const float x = key_x(kl);
        if (kl != 0ull && x != -INFINITY) cl_ = sw + ((x - hw) - lw);
      }
    } else {
      kl = 0ull;
    }
    // ---- the sentence's ranking: (score desc, list position asc) = (score desc, flat index asc)
    const int nvalid = __popc(__ballot_sync(FULL, kl != 0ull));
    {
      const int rank = warp_rank_u32(kl != 0ull ? ord_f32(cl_ + 0.0f) : 0u, lane);   // + 0: -0 ranks as +0
      if (kl != 0ull && rank < 2 * W) sh.cm_sel[rank] = lane;
    }
    sh.cm_key[lane] = kl;
    sh.cm_c[lane] = cl_;
    sh.cm_w[lane] = wl;
    __syncwarp();
    // ---- the walk, one lane per rank (2W <= 32): the k-th candidate that is not an EOS hit
    // becomes new beam k, for k < W; an EOS hit at rank < W that the walk reaches joins the
    // finished set, in rank order
    const bool have = lane < 2 * W && lane < nvalid;
    const int jw = have ? sh.cm_sel[lane] : 0;
    const u64 kw = have ? sh.cm_key[jw] : 0ull;
    const float cw = have ? sh.cm_c[jw] : -INFINITY;
    const int ww = have ? sh.cm_w[jw] : 0;
    const u32 v = key_v(kw);
    const bool eos = have && a.eos >= 0 && v == static_cast<u32>(a.eos);
    const u32 live = __ballot_sync(FULL, have && !eos);
    const int before = __popc(live & ((1u << lane) - 1u));
    const unsigned sl = __fns(live, 0, lane + 1);  // the (lane+1)-th live lane, if any
    const int src_lane = sl < 32u ? static_cast<int>(sl) : 0;
    const float c_in = __shfl_sync(FULL, cw, src_lane);
    const u32 v_in = __shfl_sync(FULL, v, src_lane);
    const int w_in = __shfl_sync(FULL, ww, src_lane);
    const int new_cnt = min(__popc(live), W);
    if (lane < new_cnt) {
      nb_score = c_in;
      nb_tok = static_cast<int>(v_in);
      nb_row = r0 + w_in;
    } else if (lane < W) {
      nb_score = -INFINITY;
    }
    const u32 hits = __ballot_sync(FULL, eos && lane < W && before < W);
    const float best = __shfl_sync(FULL, cw, 0);
    // BeamHypotheses.add for each EOS hit, in rank order (slot q lives in lane q)
    float f_ns = fns;
    int f_len = flen, f_ser = fser;
    for (u32 m = hits; m; m &= m - 1) {
      const int rank = __ffs(m) - 1;
      const float ns = __shfl_sync(FULL, cw, rank) / a.lp_tf;
      const int src = r0 + __shfl_sync(FULL, ww, rank);
      int slot = -1;
      if (fcount < W) {
        slot = fcount;
      } else if (ns > fworst) {                    // evict the worst; ties: the earliest inserted
        float bn = lane < W ? f_ns : INFINITY;
        int bs2 = lane < W ? f_ser : 0x7fffffff, bl = lane;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float on = __shfl_xor_sync(FULL, bn, off);
          const int os = __shfl_xor_sync(FULL, bs2, off);
          const int ol = __shfl_xor_sync(FULL, bl, off);
          if (on < bn || (on == bn && (os < bs2 || (os == bs2 && ol < bl)))) { bn = on; bs2 = os; bl = ol; }
        }
        slot = bl;
      }
      if (slot >= 0) {
        if (lane == slot) {
          f_ns = ns;
          f_len = t;
          f_ser = fnext;
          f_src = src;
        }
        fnext += 1;
        if (fcount < W) {
          fcount += 1;
          fworst = fminf(ns, fworst);
        }
        if (fcount >= W) {
          float wmin = lane < W ? f_ns : INFINITY;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) wmin = fminf(wmin, __shfl_xor_sync(FULL, wmin, off));
          fworst = wmin;
        }
      }
    }
    if (lane == 0 && new_cnt < W) set_status(a.status, VBS_EINPUT);
    bool done = false;
    if (fcount >= W) done = a.early_stopping == VBS_ES_TRUE || fworst >= best / a.lp_boundf;
    done_now = done ? 1 : 0;
    // the step's finished-sentence count, issued before the writes
    if (lane == 0) old_cnt = atomicAdd(reinterpret_cast<unsigned*>(a.done_count), (1u << 16) | done_now);
    if (lane < W && VBS_CHECK(r0 + lane < a.R && nb_row >= r0 && nb_row < r0 + W, 3, nb_row, a.status)) {
      a.beam_idx[r0 + lane] = nb_row;
      a.tokens[r0 + lane] = nb_tok;
      a.scores[r0 + lane] = nb_score;
      a.fin_ns[r0 + lane] = static_cast<double>(f_ns);
      a.fin_len[r0 + lane] = f_len;
      a.fin_serial[r0 + lane] = f_ser;
    }
    if (lane == 0) {
      a.fin_count[b] = fcount;
      a.fin_next[b] = fnext;
      a.fin_worst[b] = static_cast<double>(fworst);
      a.done[b] = done_now;
    }
    // the sequence gather: every thread of the CTA, from these decisions
    if (lane < W) {
      sh.cm_nbrow[lane] = nb_row;
      sh.cm_fsrc[lane] = f_src;
      sh.cm_nbtok[lane] = nb_tok;
    }
    if (lane == 0) sh.cm_gather = 1;
  } else {
    if (lane == 0) old_cnt = atomicAdd(reinterpret_cast<unsigned*>(a.done_count), (1u << 16) | 1u);
    if (lane < W) {
      a.beam_idx[r0 + lane] = -1;
      a.tokens[r0 + lane] = a.pad;
      a.scores[r0 + lane] = 0.f;
      a.seqs[static_cast<int64_t>(r0 + lane) * ld + t] = a.pad;
    }
    if (lane == 0) sh.cm_gather = 0;
  }
}

// Every thread of the cluster's first CTA, after the merge's decisions (and its prefetch of
// the first sequence columns) are visible: the parents' columns [0, t) gathered in place --
// the prefetched ones directly, the rest staged one column tile at a time through the free
// ring -- and the new token at column t; the finished hypotheses' tokens likewise.
__device__ void cluster_gather(const BsArgs& a, BsShared& sh, int b) {
  if (!sh.cm_gather) return;                       // the same for every thread
  const int W = a.W, r0 = b * W, t = a.t, ld = a.seq_ld, tid = threadIdx.x;
  int* tile = reinterpret_cast<int*>(&sh.ring[0][0]);
  const int TWp = PF_TILE / W, ncp = min(t, TWp);
  for (int i = tid; i < W * ncp; i += BS_NT) {
    const int w = i / ncp, c = i - w * ncp;
    const int pr = sh.cm_nbrow[w] - r0, fs = sh.cm_fsrc[w];
    if (!VBS_CHECK(pr >= 0 && pr < W && (fs < 0 || (fs >= r0 && fs < r0 + W)) && c < ld, 4, pr, a.status)) continue;
    a.seqs[static_cast<int64_t>(r0 + w) * ld + c] = sh.pf_tile[pr * TWp + c];
    if (fs >= 0) a.fin_tok[static_cast<int64_t>(r0 + w) * ld + c] = sh.pf_tile[(fs - r0) * TWp + c];
  }
  const int TWc = CM_TILE / W;
  for (int c0 = ncp; c0 < t; c0 += TWc) {
    const int nc = min(TWc, t - c0);
    __syncthreads();                               // the tile's previous contents are written out
    for (int i = tid; i < W * nc; i += BS_NT) {
      const int w = i / nc, c = i - w * nc;
      tile[w * TWc + c] = __ldcg(a.seqs + static_cast<int64_t>(r0 + w) * ld + c0 + c);
    }
    __syncthreads();
    for (int i = tid; i < W * nc; i += BS_NT) {
      const int w = i / nc, c = i - w * nc;
      const int pr = sh.cm_nbrow[w] - r0, fs = sh.cm_fsrc[w];
      if (!VBS_CHECK(pr >= 0 && pr < W && (fs < 0 || (fs >= r0 && fs < r0 + W)), 4, pr, a.status)) continue;
      a.seqs[static_cast<int64_t>(r0 + w) * ld + c0 + c] = tile[pr * TWc + c];
      if (fs >= 0) a.fin_tok[static_cast<int64_t>(r0 + w) * ld + c0 + c] = tile[(fs - r0) * TWc + c];
    }
  }
  if (tid < W) a.seqs[static_cast<int64_t>(r0 + tid) * ld + t] = sh.cm_nbtok[tid];
}

template <typename T, bool TMA, bool FUSE>
__global__ void __launch_bounds__(BS_NT, 1) bs_cluster_kernel(const BsArgs a) {
  extern __shared__ __align__(128) unsigned char bs_smem[];
  BsShared& sh = *reinterpret_cast<BsShared*>(bs_smem);
  const int C = a.cluster;
  const int b = static_cast<int>(blockIdx.x) / C, c = static_cast<int>(blockIdx.x) - b * C;
  const int RPC = a.W / C;
  const int64_t e0 = (static_cast<int64_t>(b) * a.W + c * RPC) * a.V;
  const int64_t e1 = e0 + static_cast<int64_t>(RPC) * a.V;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], BS_NCW);
    }
    fence_mbar_init();
  }
  if (threadIdx.x < NSLOT) {
    sh.thr[threadIdx.x] = 0u;
    sh.tmin[threadIdx.x] = 0xffffffffu;
    sh.qcnt[threadIdx.x] = 0;
    sh.qref[threadIdx.x] = 0;
    sh.mode[threadIdx.x] = 0;
  }
  for (int i = threadIdx.x; i < NSLOT * QSEG; i += BS_NT) (&sh.q[0][0])[i] = 0ull;
  __syncthreads();
  // launched as a programmatic dependent: the set-up above overlaps the previous kernel's
  // tail; every global access comes after it has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if ((threadIdx.x >> 5) == BS_NCW) {
    const int lane = threadIdx.x & 31;
    if (TMA && lane == 0) {
      produce<T>(a, sh, e0, e1);
    } else if (FUSE && c == 0) {
      // the idle producer lanes pull the sentence's KV block state into L2 for the
      // remap that follows the merge
      const PagedArgs& kv = a.kv;
      const int r0 = b * a.W;
      prefetch_l2(kv.table + static_cast<int64_t>(r0) * kv.MB, static_cast<int64_t>(a.W) * kv.MB * 4, lane - 1, 31);
      prefetch_l2(kv.refcnt + static_cast<int64_t>(b) * kv.S, static_cast<int64_t>(kv.S) * 4, lane - 1, 31);
      prefetch_l2(kv.stack + static_cast<int64_t>(b) * kv.S, static_cast<int64_t>(kv.S) * 4, lane - 1, 31);
      prefetch_l2(kv.nblk + r0, static_cast<int64_t>(a.W) * 4, lane - 1, 31);
      prefetch_l2(kv.top + b, 4, lane - 1, 31);
    }
  } else {
    if (c == 0 && threadIdx.x < 32) cluster_prefetch(a, sh, b, threadIdx.x);
    consume<T, TMA, false>(a, sh, e0, e1);
  }
  __syncwarp();
  cooperative_groups::this_cluster().sync();       // every CTA's row results are in its shared memory
  if (c == 0) {
    unsigned old_cnt = 0;
    int done_now = 0;
    if (threadIdx.x < 32) cluster_merge_sentence(a, sh, b, threadIdx.x, old_cnt, done_now);
    __syncthreads();                               // the decisions, for the gather by every thread
    cluster_gather(a, sh, b);
    // the last sentence of the step reports whether all are finished
    if (threadIdx.x == 0 && (old_cnt >> 16) == static_cast<unsigned>(a.B - 1)) {
      const int all = static_cast<int>((old_cnt & 0xffffu) + done_now) == a.B;
      *a.all_done_dev = all;
      if (a.all_done_out) *a.all_done_out = all;
      *a.done_count = 0;
    }
  }
  cooperative_groups::this_cluster().sync();       // keep them readable until the merge is done
  if (FUSE && c == 0) {
    // the paged KV remap of the sentence, on the step's beam_idx just written; the ring is
    // free now and holds its shared state
    RemapShared& rsh = *reinterpret_cast<RemapShared*>(&sh.ring[0][0]);
    int32_t* rs = reinterpret_cast<int32_t*>(&sh.ring[0][0] + REMAP_SH_BYTES);
    paged_remap_sentence<BS_NT>(a.kv, b, a.beam_idx, a.kv_t, rs, rsh);
  }
}

// ---------------------------------------------------------------------------------------
// the merge kernel: one CTA per sentence
// ---------------------------------------------------------------------------------------

// All threads: one round of independent loads of sentence b's rows' partial slots (all P
// of them; the merge uses the first np).  P * K <= PART_KEYS and W * P <= PART_KEYS / 2.
__device__ void merge_prefetch_partials(const BsArgs& a, MergeShared& sm, int b, int nthreads) {
  const int W = a.W, K = a.K, P = a.P;
  const int r0 = b * W;
  const int PK = P * K;
  const u64* keys = a.part_key + static_cast<int64_t>(r0) * PK;
  for (int f = threadIdx.x; f < W * PK; f += nthreads) {
    const int w = f / PK;
    sm.rowscratch[w * PART_KEYS + (f - w * PK)] = __ldcg(keys + f);
  }
  for (int f = threadIdx.x; f < W * P; f += nthreads) {
    sm.pM[f] = __ldcg(a.part_M + static_cast<int64_t>(r0) * P + f);
    sm.pL[f] = __ldcg(a.part_l + static_cast<int64_t>(r0) * P + f);
  }
}

// Sentence b's rows' scores and partial counts (neither is written by the stream kernel).
__device__ void merge_prefetch_rows(const BsArgs& a, MergeShared& sm, int b) {
  const int r0 = b * a.W;
  if (threadIdx.x < a.W) {
    sm.s[threadIdx.x] = __ldcg(a.scores + r0 + threadIdx.x);
    sm.np[threadIdx.x] = a.row_np[r0 + threadIdx.x];
  }
}



// Warp-wide, from the prefetched partials: row w's LSE (split hi + lo in fp32) and its
// sorted top-K list with scores.
__device__ void row_merge(const BsArgs& a, MergeShared& sm, int w, int lane) {
  const int K = a.K;
  const float s = sm.s[w];
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
  const int n = sm.np[w];
  const u64* scratch = sm.rowscratch + w * PART_KEYS;
  float Mc = -INFINITY, lc = 0.f;
  for (int c = lane; c < n; c += 32) lse_merge(Mc, lc, sm.pM[w * a.P + c], sm.pL[w * a.P + c]);
  for (int off = 1; off < n && off < 32; off <<= 1) {      // lanes >= n hold (-inf, 0)
    const float M2 = __shfl_xor_sync(FULL, Mc, off);
    const float l2 = __shfl_xor_sync(FULL, lc, off);
    lse_merge(Mc, lc, M2, l2);
  }
  Mc = __shfl_sync(FULL, Mc, 0);
  lc = __shfl_sync(FULL, lc, 0);
  u64* out = sm.wtop + w * K;
  if (n == 1) {
    if (lane < K) out[lane] = scratch[lane];
    __syncwarp();
  } else if (8 * (n - 1) < 5 * K) {
    // few lists of many keys: fold them pairwise, 32 best at a time (lanes >= K hold 0)
    u64 cur = lane < K ? scratch[lane] : 0ull;
    for (int j = 1; j < n; ++j) cur = warp_merge_top32(cur, lane < K ? scratch[j * K + lane] : 0ull, lane);
    if (lane < K) out[lane] = cur;
    __syncwarp();
  } else {
    warp_merge_sorted(scratch, n, K, out, lane);
  }
  // LSE = ln2 * (Mc + log2 lc) as an unevaluated fp32 sum hi + lo (error-free sum and
  // product steps; FP64 is slow on this part and not needed)
  const float L2 = log2f(lc);
  const float t_hi = Mc + L2;
  const float bb = t_hi - Mc;
  const float t_lo = (Mc - (t_hi - bb)) + (L2 - bb);
  const float p = t_hi * LN2_HI;
  const float e = fmaf(t_hi, LN2_HI, -p) + fmaf(t_hi, LN2_LO, t_lo * LN2_HI);
  const float hi = p + e;
  const float lo = e - (hi - p);
  if (lane == 0 && !(hi > -INFINITY && hi < INFINITY)) set_status(a.status, VBS_EINPUT);  // no finite logit, NaN, +inf
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

// A CTA's barrier: __syncthreads (BAR = 0) or named barrier BAR among the first NT threads.
template <int NT, int BAR>
__device__ __forceinline__ void cta_sync() {
  if constexpr (BAR == 0) __syncthreads();
  else named_sync(BAR, NT);
}

// Threads 0..NT-1, sentence b: the inputs earlier kernels wrote -- the sentence state, the
// rows' scores and partial counts, the first tile of the parents' sequences -- into shared
// memory; returns the sentence's done flag.
template <int NT>
__device__ int merge_load_state(const BsArgs& a, MergeShared& sm, int b) {
  const int tid = threadIdx.x;
  const int W = a.W, r0 = b * W, t = a.t, ld = a.seq_ld;
  const int TW = SEQ_TILE_INTS / W;
  const int nc0 = min(t, TW);
  const int done_b = __ldcg(a.done + b);
  merge_prefetch_rows(a, sm, b);
  // all through L2: earlier steps wrote them from other SMs
  for (int i = tid; i < W * nc0; i += NT) {
    const int w = i / nc0, c = i - w * nc0;
    sm.tile[w * TW + c] = __ldcg(a.seqs + static_cast<int64_t>(r0 + w) * ld + c);
  }
  if (tid < W) {
    sm.f_ns[tid] = static_cast<float>(__ldcg(a.fin_ns + r0 + tid));
    sm.f_len[tid] = __ldcg(a.fin_len + r0 + tid);
    sm.f_serial[tid] = __ldcg(a.fin_serial + r0 + tid);
    sm.f_src[tid] = -1;
  }
  if (tid == 0) {
    sm.f_count = __ldcg(a.fin_count + b);
    sm.f_next = __ldcg(a.fin_next + b);
    sm.f_worst = static_cast<float>(__ldcg(a.fin_worst + b));
  }
  return done_b;
}

// Threads 0..NT-1 (NT a multiple of 32; the warps take the rows in turn): sentence b's merge
// once its state and partials are in shared memory (the caller's barrier has passed): row
// LSEs and lists, the ranking by (score desc, flat index asc), the walk with
// BeamHypotheses.add, the stopping test, the outputs and the in-place sequence gather.
template <int NT, int BAR>
__device__ void merge_sentence(const BsArgs& a, MergeShared& sm, int b, int done_b) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int W = a.W, K = a.K;
  const int r0 = b * W;
  const int t = a.t;
  const int ld = a.seq_ld;
  const int TW = SEQ_TILE_INTS / W;            // columns per row in one gather tile
  const bool was_done = done_b != 0;
  if (!was_done)
    for (int w = warp; w < W; w += NW) row_merge(a, sm, w, lane);
  cta_sync<NT, BAR>();

  if (!was_done && W * K <= 32) {
    // one warp ranks every candidate by (score desc, flat index asc): list position f =
    // w*K + i grows with the flat index, and invalid entries (0) rank last
    if (warp == 0) {
      const int w = lane / K, i = lane - w * K;
      const bool valid = lane < W * K && i < sm.nval[w];
      const float c = valid ? sm.candv[lane] : -INFINITY;
      const int rank = warp_rank_u32(valid ? ord_f32(c + 0.0f) : 0u, lane);   // + 0: -0 ranks as +0
      if (valid && rank < 2 * W) {
        sm.sel_w[rank] = w;
        sm.sel_i[rank] = i;
        sm.sel_c[rank] = c;
      }
    }
  } else if (!was_done) {
    // the W lists as keys (score desc, then row and list position asc -- the flat index
    // order), merged pairwise, 32 best at a time, level by level across the warps (2W <= 32);
    // the rows' partial lists are consumed, so their scratch holds the levels
    u64* lev = sm.rowscratch;
    const auto row_key = [&](int w) -> u64 {
      if (w >= W || lane >= K || lane >= sm.nval[w]) return 0ull;
      return (static_cast<u64>(ord_f32(sm.candv[w * K + lane] + 0.0f)) << 32) |   // + 0: -0 ranks as +0
             static_cast<u64>(~static_cast<u32>((w << 8) | lane));
    };
    int m = (W + 1) / 2, src = 0;
    for (int p = warp; p < m; p += NW) {
      const u64 r = warp_merge_top32(row_key(2 * p), row_key(2 * p + 1), lane);
      lev[p * 32 + lane] = r;
    }
    cta_sync<NT, BAR>();
    while (m > 1) {
      const int m2 = (m + 1) / 2, dst = src ^ 1;
      for (int p = warp; p < m2; p += NW) {
        const u64 a0 = lev[src * 512 + (2 * p) * 32 + lane];
        const u64 b0 = 2 * p + 1 < m ? lev[src * 512 + (2 * p + 1) * 32 + lane] : 0ull;
        lev[dst * 512 + p * 32 + lane] = warp_merge_top32(a0, b0, lane);
      }
      cta_sync<NT, BAR>();
      m = m2;
      src = dst;
    }
    if (tid < 2 * W) {
      const u64 k = lev[src * 512 + tid];
      if (k != 0ull) {
        const u32 lo = ~static_cast<u32>(k);
        sm.sel_w[tid] = static_cast<int>(lo >> 8);
        sm.sel_i[tid] = static_cast<int>(lo & 0xffu);
        sm.sel_c[tid] = unord_f32(static_cast<u32>(k >> 32));
      }
    }
  }
  cta_sync<NT, BAR>();

  if (warp == 0 && !was_done) {
    // The walk of the ranked candidates, one lane per rank (2W <= 32): the k-th candidate
    // that is not an EOS hit becomes new beam k, for k < W; an EOS hit at rank < W that
    // the walk reaches (fewer than W live candidates before it) joins the finished set,
    // in rank order.
    int nv = lane < W ? sm.nval[lane] : 0;
    nv = __reduce_add_sync(FULL, nv);
    const bool have = lane < 2 * W && lane < nv;
    int w = 0;
    float c = -INFINITY;
    u32 v = 0;
    if (have) {
      w = sm.sel_w[lane];
      c = sm.sel_c[lane];
      v = key_v(sm.wtop[w * K + sm.sel_i[lane]]);
    }
    const bool eos = have && a.eos >= 0 && v == static_cast<u32>(a.eos);
    const u32 live = __ballot_sync(FULL, have && !eos);
    const int before = __popc(live & ((1u << lane) - 1u));
    if (have && !eos && before < W) {
      sm.nb_score[before] = c;
      sm.nb_tok[before] = static_cast<int>(v);
      sm.nb_row[before] = r0 + w;
    }
    const u32 hits = __ballot_sync(FULL, eos && lane < W && before < W);
    const int new_cnt = min(__popc(live), W);
    if (lane == 0) {
      const float lp_t = a.lp_tf;
      for (u32 m = hits; m; m &= m - 1) {
        const int rank = __ffs(m) - 1;
        // BeamHypotheses.add(hyp = the parent's sequence, sum = c), |y| = t
        const float ns = sm.sel_c[rank] / lp_t;
        int slot = -1;
        if (sm.f_count < W) {
          slot = sm.f_count++;
          sm.f_worst = fminf(ns, sm.f_worst);
        } else if (ns > sm.f_worst) {
          slot = 0;                            // evict the worst; ties: the earliest inserted
          for (int q = 1; q < W; ++q)
            if (sm.f_ns[q] < sm.f_ns[slot] || (sm.f_ns[q] == sm.f_ns[slot] && sm.f_serial[q] < sm.f_serial[slot]))
              slot = q;
        }
        if (slot >= 0) {
          sm.f_ns[slot] = ns;
          sm.f_len[slot] = t;
          sm.f_serial[slot] = sm.f_next++;
          sm.f_src[slot] = r0 + sm.sel_w[rank];
          if (sm.f_count >= W) {
            float wmin = sm.f_ns[0];
            for (int q = 1; q < W; ++q) wmin = fminf(wmin, sm.f_ns[q]);
            sm.f_worst = wmin;
          }
        }
      }
      if (new_cnt < W) set_status(a.status, VBS_EINPUT);
      for (int q = new_cnt; q < W; ++q) { sm.nb_score[q] = -INFINITY; sm.nb_tok[q] = a.pad; sm.nb_row[q] = r0; }
      bool done = false;
      if (sm.f_count >= W)
        done = a.early_stopping == VBS_ES_TRUE || sm.f_worst >= sm.sel_c[0] / a.lp_boundf;
      sm.done_now = done ? 1 : 0;
    }
  }
  if (tid == 0 && was_done) sm.done_now = 1;
  cta_sync<NT, BAR>();

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
      a.fin_ns[r0 + tid] = static_cast<double>(sm.f_ns[tid]);
      a.fin_len[r0 + tid] = sm.f_len[tid];
      a.fin_serial[r0 + tid] = sm.f_serial[tid];
    }
    if (tid == 0) {
      a.fin_count[b] = sm.f_count;
      a.fin_next[b] = sm.f_next;
      a.fin_worst[b] = static_cast<double>(sm.f_worst);
      a.done[b] = sm.done_now;
    }
    // sequences: gather the parents' columns [0, t) in place (tile 0 is prefetched), append the token
    for (int c0 = 0; c0 < t; c0 += TW) {
      const int nc = min(TW, t - c0);
      if (c0 > 0) {
        cta_sync<NT, BAR>();
        for (int i = tid; i < W * nc; i += NT) {
          const int w = i / nc, c = i - w * nc;
          sm.tile[w * TW + c] = __ldcg(a.seqs + static_cast<int64_t>(r0 + w) * ld + c0 + c);
        }
        cta_sync<NT, BAR>();
      }
      for (int i = tid; i < W * nc; i += NT) {
        const int w = i / nc, c = i - w * nc;
        if (!VBS_CHECK(sm.nb_row[w] >= r0 && sm.nb_row[w] < r0 + W &&
                           (sm.f_src[w] < 0 || (sm.f_src[w] >= r0 && sm.f_src[w] < r0 + W)), 5, sm.nb_row[w], a.status))
          continue;
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

__global__ void __launch_bounds__(MG_NT) bs_merge_kernel(const BsArgs a) {
  extern __shared__ __align__(16) unsigned char mg_smem[];
  MergeShared& sm = *reinterpret_cast<MergeShared*>(mg_smem);
  const int b = blockIdx.x;
  // The stream kernel writes only the partials.  It starts after every earlier kernel on
  // the stream has finished, so the sentence state, scores and sequences can load while
  // it runs; the partials load after griddepcontrol.wait.
  const int done_b = merge_load_state<MG_NT>(a, sm, b);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  merge_prefetch_partials(a, sm, b, MG_NT);
  __syncthreads();
  merge_sentence<MG_NT, 0>(a, sm, b, done_b);
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
__global__ void bs_finalize_kernel(const BsArgs a, const float* scores, const int32_t* seqs, int n_ret,
                                   int32_t* out_seqs, int32_t* out_len, float* out_score) {
  __shared__ double f_ns[WMAX];
  __shared__ int f_serial[WMAX], f_src[WMAX], f_ntok[WMAX];
  __shared__ int s_order[WMAX];
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
    // the n_ret best by (normalised score desc, insertion order desc): the j-th takes the best
    // of the slots not yet taken
    unsigned taken = 0u;
    for (int j = 0; j < n_ret; ++j) {
      int best = -1;
      for (int q = 0; q < count; ++q) {
        if (taken >> q & 1u) continue;
        if (best < 0 || f_ns[q] > f_ns[best] || (f_ns[q] == f_ns[best] && f_serial[q] > f_serial[best])) best = q;
      }
      if (best < 0) best = 0;                         // fewer hypotheses than n_ret: never with n_ret <= W
      taken |= 1u << best;
      s_order[j] = best;
      const int row = b * n_ret + j;
      out_score[row] = static_cast<float>(f_ns[best]);
      const int n = f_ntok[best];
      out_len[row] = (n < ld && a.eos >= 0) ? n + 1 : n;
    }
  }
  __syncthreads();
  for (int j = 0; j < n_ret; ++j) {
    const int q = s_order[j];
    const int n = f_ntok[q];
    if (!VBS_CHECK(f_src[q] < a.R && q < W, 6, f_src[q], a.status)) continue;
    const int32_t* src = f_src[q] >= 0 ? seqs + static_cast<int64_t>(f_src[q]) * ld
                                       : a.fin_tok + static_cast<int64_t>(r0 + q) * ld;
    int32_t* dst = out_seqs + (static_cast<int64_t>(b) * n_ret + j) * ld;
    for (int c = threadIdx.x; c < ld; c += blockDim.x) {
      int v = a.pad;
      if (c < n) v = src[c];
      else if (c == n && a.eos >= 0) v = a.eos;
      dst[c] = v;
    }
  }
}

// ---------------------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------------------

template <typename T, bool TMA, bool BIGK>
static int launch_stream_k(const BsArgs& a, int grid, cudaStream_t s) {
  static std::atomic<unsigned long long> attr_done{0};
  const int smem = static_cast<int>(sizeof(BsShared));
  if (!smem_attr_once(bs_stream_kernel<T, TMA, BIGK>, smem, attr_done)) return VBS_ECUDA;
  bs_stream_kernel<T, TMA, BIGK><<<grid, BS_NT, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

// K > 8 (W > 4) takes the instance with the cross-warp seed and exact queue bars; the
// smaller lists keep the lighter loop.
template <typename T, bool TMA>
static int launch_stream(const BsArgs& a, int grid, cudaStream_t s) {
  return a.K > 8 ? launch_stream_k<T, TMA, true>(a, grid, s) : launch_stream_k<T, TMA, false>(a, grid, s);
}

// The merge grid is a programmatic dependent of the stream grid: it may launch
// while the stream CTAs retire and waits for their writes in griddepcontrol.wait.
static int launch_merge(const BsArgs& a, cudaStream_t s) {
  static std::atomic<unsigned long long> attr_done{0};
  const int smem = static_cast<int>(sizeof(MergeShared));
  if (!smem_attr_once(bs_merge_kernel, smem, attr_done)) return VBS_ECUDA;
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

template <typename T, bool TMA, bool FUSE>
static int launch_cluster(const BsArgs& a, cudaStream_t s) {
  static std::atomic<unsigned long long> attr_done{0};
  const int smem = static_cast<int>(sizeof(BsShared));
  if (!smem_attr_once(bs_cluster_kernel<T, TMA, FUSE>, smem, attr_done)) return VBS_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.cluster);
  cfg.blockDim = dim3(BS_NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, bs_cluster_kernel<T, TMA, FUSE>, a) == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

// ---------------------------------------------------------------------------------------
// ablation: the two-pass coarse selection of the pages' LightSeq article (R-top-k)
// ---------------------------------------------------------------------------------------
//
// The article's first pass over a row splits its logits into K groups, takes each group's
// maximum and the smallest of those maxima, R (at most the row's K-th largest logit: the
// K maxima are K distinct logits at or above R), together with the row's log-sum-exp;
// the second pass reads the row again and queues every logit >= R; a sort of the queue
// gives the exact top K.  Here the groups are the logits each thread reads, grouped by
// thread index mod K (any split into K non-empty groups bounds the K-th largest; an empty
// group makes R the lowest bar), the queue keeps the row's K best keys exactly (a pass that
// overflows raises the bar to the K-th best key it holds, which only rises, and runs
// again), and each row's (max, scaled sum, K best keys) goes to the partial slot the merge
// kernel reads, so the rest of the step is the two-kernel path's merge.  The logits are
// read twice: the path exists to measure that against the one-pass kernels.

constexpr int RT_NT = 256;
constexpr int RT_U = 4;
constexpr int RT_CAP = 2048;

template <typename T, bool VECTOR>
__global__ void __launch_bounds__(RT_NT) rtopk_pass1_kernel(const BsArgs a) {
  constexpr int VEC = VECTOR ? Vec16<T>::N : 1;
  __shared__ float sM[RT_NT / 32], sl[RT_NT / 32];
  __shared__ u32 gmax[KMAX];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  if (tid < K) gmax[tid] = 0u;
  __syncthreads();
  if (row_skipped(a, r)) return;                    // the same for every thread of the row
  const char* row = reinterpret_cast<const char*>(a.logits) + static_cast<int64_t>(r) * a.ld * Elem<T>::BYTES;
  const int n = a.V / VEC;
  float m = -INFINITY, M = -INFINITY, l = 0.f;
  for (int i0 = tid; i0 < n; i0 += RT_NT * RT_U) {
    float x[RT_U][VEC];
#pragma unroll
    for (int u = 0; u < RT_U; ++u) {
      const int i = i0 + u * RT_NT;
      if (i < n) {
        if constexpr (VECTOR) Vec16<T>::unpack(ld_stream16(row + static_cast<int64_t>(i) * 16), x[u]);
        else x[u][0] = Elem<T>::load(row, i);
      } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) x[u][e] = -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < RT_U; ++u) {
      float tm = x[u][0];
#pragma unroll
      for (int e = 1; e < VEC; ++e) tm = fmaxf(tm, x[u][e]);
      if (tm > m) {
        const float Mn = tm * LOG2E_F;
        l *= ex2(M - Mn);
        M = Mn;
        m = tm;
      }
      if (tm > -INFINITY) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) l += ex2(fmaf(x[u][e], LOG2E_F, -M));
      }
    }
  }
  if (m > -INFINITY) atomicMax(&gmax[tid % K], ord_f32(m));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float M2 = __shfl_xor_sync(FULL, M, off);
    const float l2 = __shfl_xor_sync(FULL, l, off);
    lse_merge(M, l, M2, l2);
  }
  if (lane == 0) { sM[warp] = M; sl[warp] = l; }
  __syncthreads();
  if (warp == 0) {
    M = lane < RT_NT / 32 ? sM[lane] : -INFINITY;
    l = lane < RT_NT / 32 ? sl[lane] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float M2 = __shfl_xor_sync(FULL, M, off);
      const float l2 = __shfl_xor_sync(FULL, l, off);
      lse_merge(M, l, M2, l2);
    }
    if (lane == 0) {
      const int64_t slot = static_cast<int64_t>(r) * a.P;
      a.part_M[slot] = M;
      a.part_l[slot] = l;
      u32 rb = gmax[0];
      for (int g = 1; g < K; ++g) rb = min(rb, gmax[g]);
      a.rtopk_bar[r] = rb;
    }
  }
}

template <typename T, bool VECTOR>
__global__ void __launch_bounds__(RT_NT) rtopk_pass2_kernel(const BsArgs a) {
  constexpr int VEC = VECTOR ? Vec16<T>::N : 1;
  __shared__ u64 q[RT_CAP];
  __shared__ u64 sel[KMAX];
  __shared__ u64 bar;
  __shared__ int cnt;
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  if (row_skipped(a, r)) return;
  const char* row = reinterpret_cast<const char*>(a.logits) + static_cast<int64_t>(r) * a.ld * Elem<T>::BYTES;
  const int n = a.V / VEC;
  if (tid == 0) bar = static_cast<u64>(a.rtopk_bar[r]) << 32;
  for (;;) {
    if (tid == 0) cnt = 0;
    __syncthreads();
    const u64 b = bar;
    for (int i0 = tid; i0 < n; i0 += RT_NT * RT_U) {
      float x[RT_U][VEC];
#pragma unroll
      for (int u = 0; u < RT_U; ++u) {
        const int i = i0 + u * RT_NT;
        if (i < n) {
          if constexpr (VECTOR) Vec16<T>::unpack(ld_stream16(row + static_cast<int64_t>(i) * 16), x[u]);
          else x[u][0] = Elem<T>::load(row, i);
        }
      }
#pragma unroll
      for (int u = 0; u < RT_U; ++u) {
        const int i = i0 + u * RT_NT;
        if (i >= n) continue;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const u64 key = make_key(x[u][e], static_cast<u32>(a.vbase + i * VEC + e));
          if (key >= b) {
            const int pos = atomicAdd(&cnt, 1);
            if (pos < RT_CAP) q[pos] = key;
          }
        }
      }
    }
    __threadfence_block();
    __syncthreads();
    const int c = cnt;
    __syncthreads();                                // every thread has read the count
    if (c <= RT_CAP) break;                         // the same for every thread
    if (warp == 0) {
      warp_select_topk(q, RT_CAP, K, sel, lane);
      if (lane == 0) bar = sel[K - 1];
    }
    __syncthreads();
  }
  // the count is read again here, after the second barrier: a selection over the count read
  // right after the collection barrier was seen, in two builds, to miss one key a lane of
  // warp 0 had queued; with the count read here no miss has been seen
  if (warp == 0) {
    warp_select_topk(q, min(*reinterpret_cast<volatile int*>(&cnt), RT_CAP), K, sel, lane);
    if (lane < K) a.part_key[static_cast<int64_t>(r) * a.P * K + lane] = sel[lane];
  }
}

int launch_bs_step_two_pass(const BsArgs& a0, bool vector_ok, cudaStream_t s) {
  BsArgs a = a0;
  a.row_np = a.row_one;                             // one partial slot per row
  if (a.dtype == VBS_BF16) {
    if (vector_ok) {
      rtopk_pass1_kernel<bf16_t, true><<<a.R, RT_NT, 0, s>>>(a);
      rtopk_pass2_kernel<bf16_t, true><<<a.R, RT_NT, 0, s>>>(a);
    } else {
      rtopk_pass1_kernel<bf16_t, false><<<a.R, RT_NT, 0, s>>>(a);
      rtopk_pass2_kernel<bf16_t, false><<<a.R, RT_NT, 0, s>>>(a);
    }
  } else {
    if (vector_ok) {
      rtopk_pass1_kernel<float, true><<<a.R, RT_NT, 0, s>>>(a);
      rtopk_pass2_kernel<float, true><<<a.R, RT_NT, 0, s>>>(a);
    } else {
      rtopk_pass1_kernel<float, false><<<a.R, RT_NT, 0, s>>>(a);
      rtopk_pass2_kernel<float, false><<<a.R, RT_NT, 0, s>>>(a);
    }
  }
  if (cudaGetLastError() != cudaSuccess) return VBS_ECUDA;
  return launch_merge(a, s);
}

// ---------------------------------------------------------------------------------------
// vocabulary shards: each shard's rows reduce to a partial with the two passes above (token
// ids offset by the shard's first column), and the merge kernel combines the shards'
// partials as it combines the stream kernel's, with the shards as a row's partial slots
// ---------------------------------------------------------------------------------------

void shard_partial_layout(int R, int K, size_t* off_l, size_t* off_key, size_t* bytes) {
  const size_t a = (static_cast<size_t>(R) * 4 + 15) / 16 * 16;
  *off_l = a;
  *off_key = 2 * a;
  *bytes = 2 * a + static_cast<size_t>(R) * K * 8;
}

int launch_bs_shard_partial(const BsArgs& a0, bool vector_ok, void* partial, cudaStream_t s) {
  size_t off_l, off_key, bytes;
  shard_partial_layout(a0.R, a0.K, &off_l, &off_key, &bytes);
  BsArgs a = a0;
  a.P = 1;                                          // one slot per row, in the caller's buffer
  a.part_M = static_cast<float*>(partial);
  a.part_l = reinterpret_cast<float*>(static_cast<char*>(partial) + off_l);
  a.part_key = reinterpret_cast<u64*>(static_cast<char*>(partial) + off_key);
  if (a.dtype == VBS_BF16) {
    if (vector_ok) {
      rtopk_pass1_kernel<bf16_t, true><<<a.R, RT_NT, 0, s>>>(a);
      rtopk_pass2_kernel<bf16_t, true><<<a.R, RT_NT, 0, s>>>(a);
    } else {
      rtopk_pass1_kernel<bf16_t, false><<<a.R, RT_NT, 0, s>>>(a);
      rtopk_pass2_kernel<bf16_t, false><<<a.R, RT_NT, 0, s>>>(a);
    }
  } else {
    if (vector_ok) {
      rtopk_pass1_kernel<float, true><<<a.R, RT_NT, 0, s>>>(a);
      rtopk_pass2_kernel<float, true><<<a.R, RT_NT, 0, s>>>(a);
    } else {
      rtopk_pass1_kernel<float, false><<<a.R, RT_NT, 0, s>>>(a);
      rtopk_pass2_kernel<float, false><<<a.R, RT_NT, 0, s>>>(a);
    }
  }
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

// One warp per row: shard j's partial of row r goes to slot r * n + j.
__global__ void bs_shard_scatter_kernel(const BsArgs a, int n, const char* partials, size_t off_l, size_t off_key,
                                        size_t bytes) {
  const int r = blockIdx.x, lane = threadIdx.x;
  const int K = a.K;
  for (int j = 0; j < n; ++j) {
    const char* p = partials + static_cast<size_t>(j) * bytes;
    const int64_t slot = static_cast<int64_t>(r) * n + j;
    if (lane == 0) {
      a.shard_M[slot] = reinterpret_cast<const float*>(p)[r];
      a.shard_l[slot] = reinterpret_cast<const float*>(p + off_l)[r];
    }
    if (lane < K) a.shard_key[slot * K + lane] = reinterpret_cast<const u64*>(p + off_key)[static_cast<int64_t>(r) * K + lane];
  }
  if (lane == 0) a.row_ns[r] = n;
}

int launch_bs_merge_shards(const BsArgs& a0, int n_shards, const void* partials, cudaStream_t s) {
  size_t off_l, off_key, bytes;
  shard_partial_layout(a0.R, a0.K, &off_l, &off_key, &bytes);
  bs_shard_scatter_kernel<<<a0.R, 32, 0, s>>>(a0, n_shards, static_cast<const char*>(partials), off_l, off_key,
                                               bytes);
  if (cudaGetLastError() != cudaSuccess) return VBS_ECUDA;
  BsArgs a = a0;
  a.P = n_shards;
  a.part_M = a.shard_M;
  a.part_l = a.shard_l;
  a.part_key = a.shard_key;
  a.row_np = a.row_ns;
  return launch_merge(a, s);
}

int launch_bs_step(const BsArgs& a, int grid, bool vector_ok, cudaStream_t s) {
  if (a.cluster) {
    if (a.kv_fuse) {
      if (a.dtype == VBS_BF16)
        return vector_ok ? launch_cluster<bf16_t, true, true>(a, s) : launch_cluster<bf16_t, false, true>(a, s);
      return vector_ok ? launch_cluster<float, true, true>(a, s) : launch_cluster<float, false, true>(a, s);
    }
    if (a.dtype == VBS_BF16)
      return vector_ok ? launch_cluster<bf16_t, true, false>(a, s) : launch_cluster<bf16_t, false, false>(a, s);
    return vector_ok ? launch_cluster<float, true, false>(a, s) : launch_cluster<float, false, false>(a, s);
  }
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

int launch_bs_finalize(const BsArgs& a, const float* scores, const int32_t* seqs, int n_ret, int32_t* out_seqs,
                       int32_t* out_len, float* out_score, cudaStream_t s) {
  bs_finalize_kernel<<<a.B, 128, 0, s>>>(a, scores, seqs, n_ret, out_seqs, out_len, out_score);
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

int bs_threads_per_cta() { return BS_NT; }
unsigned long long bs_check_record() { return read_check_record(); }
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
  merge_prefetch_rows(a, sm, blockIdx.x);
  merge_prefetch_partials(a, sm, blockIdx.x, MG_NT);
  __syncthreads();
  for (int w = warp; w < W; w += MG_NW) row_merge(a, sm, w, lane);
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

  static std::atomic<unsigned long long> attr_done{0};
  const int smem = static_cast<int>(sizeof(MergeShared));
  if (!smem_attr_once(bs_expand_merge_kernel, smem, attr_done)) return VBS_ECUDA;
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
