// Blockwise parallel decoding: predict (per-head argmax) and verify + accept
// (sm_103a).
//
// What is computed follows "Blockwise Parallel Decoding for Deep Autoregressive
// Models" (papercache notes), §3 (predict, verify: the largest khat such that
// every proposal up to khat equals the base model's argmax given the proposals
// before it; khat >= 1; accept) and §4 (the combined scoring and proposal model:
// the verify call also yields the next iteration's proposals from position
// khat), and §5 (approximate inference: the top-k and distance tests and the
// minimum block, whose formulas the pages' text lacks; the readings are stated at
// bpd_verify_approx).  Layout: logits[b, p, h, :] is head h+1 at proposal
// position p+1.
//
// The verify checks are sequential (each decides whether the next row is
// needed), so only the rows the definition needs are read: head 0 at positions
// 0..khat-1 (at most k-1 of them), then the k heads at position khat-1, the
// already-known head 0 reused.  Batches up to 16384 run as a persistent work
// queue (chains first, then the published head rows); larger ones one CTA per
// batch element.  Argmax ties go to the lower token id, through a (logit, token)
// key where a larger key is better.

#include "common.cuh"
#include "bs_internal.h"

namespace vbs {

constexpr int BPD_NT = 512;
constexpr int BPD_NW = BPD_NT / 32;
constexpr int BPD_U = 8;

// The verify test of one proposal (§3, or the relaxed tests of §5): exact match with
// the argmax; rank (keys above the proposal's, ties to the lower id) below crit.param;
// or a token distance |proposal - argmax| of at most crit.param.
__device__ __forceinline__ bool bpd_passes(const BpdCrit& crit, int prop, int am, int rank, int V) {
  if (crit.mode == VBS_BPD_TOPK) return prop >= 0 && prop < V && rank < crit.param;
  if (crit.mode == VBS_BPD_DISTANCE) return abs(prop - am) <= crit.param;
  return prop == am;
}

// The logit of token `tok` in a row (any value for a token outside [0, V), which passes
// no rank test).
template <typename T>
__device__ __forceinline__ float token_value(const char* row, int tok, int V) {
  return (tok >= 0 && tok < V) ? Elem<T>::load(row, tok) : 0.f;
}

// Whether element (x, v) ranks above the proposal (xp, prop): a larger logit, or an equal
// one at a lower id.
__device__ __forceinline__ int beats(float x, int v, float xp, int prop) {
  return (x > xp || (x == xp && v < prop)) ? 1 : 0;
}

// Best key of the vectors [i0, i1) of one row, for this thread (strided by `stride`);
// with RANK, *cnt also counts this thread's elements that beat the proposal (xp, prop).
template <typename T, bool VECTOR, bool RANK = false>
__device__ __forceinline__ u64 thread_row_best(const char* row, int64_t i0, int64_t i1, int64_t stride,
                                               float xp = 0.f, int prop = -1, int* cnt = nullptr) {
  constexpr int VEC = VECTOR ? Vec16<T>::N : 1;
  u64 best = 0;
  int c = 0;
  for (int64_t base = i0; base < i1; base += stride * BPD_U) {
    uint4 q[BPD_U];
    float xs[BPD_U];
#pragma unroll
    for (int u = 0; u < BPD_U; ++u) {
      int64_t i = base + u * stride;
      if (i < i1) {
        if constexpr (VECTOR) q[u] = ld_stream16(row + i * 16);
        else xs[u] = Elem<T>::load(row, i);
      }
    }
#pragma unroll
    for (int u = 0; u < BPD_U; ++u) {
      int64_t i = base + u * stride;
      if (i < i1) {
        float x[VEC];
        if constexpr (VECTOR) Vec16<T>::unpack(q[u], x);
        else x[0] = xs[u];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          u64 k = make_key(x[e], static_cast<u32>(i * VEC + e));
          best = k > best ? k : best;
          if constexpr (RANK) c += beats(x[e], static_cast<int>(i * VEC + e), xp, prop);
        }
      }
    }
  }
  if constexpr (RANK) *cnt = c;
  return best;
}

// The row's argmax; with RANK also *rank = the number of elements that beat the proposal
// (xp, prop) (every thread).
template <typename T, bool VECTOR, bool RANK = false>
__device__ __forceinline__ int cta_row_argmax(const char* row, int64_t nvec, u64* red, int* redc, float xp = 0.f,
                                              int prop = -1, int* rank = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int c = 0;
  u64 k = thread_row_best<T, VECTOR, RANK>(row, tid, nvec, BPD_NT, xp, prop, &c);
  k = warp_max_u64(k);
  if constexpr (RANK) c = __reduce_add_sync(FULL, c);
  if (lane == 0) {
    red[warp] = k;
    if constexpr (RANK) redc[warp] = c;
  }
  __syncthreads();
  if (warp == 0) {
    u64 v = lane < BPD_NW ? red[lane] : 0ull;
    v = warp_max_u64(v);
    if constexpr (RANK) {
      const int cc = __reduce_add_sync(FULL, lane < BPD_NW ? redc[lane] : 0);
      if (lane == 0) redc[BPD_NW] = cc;
    }
    if (lane == 0) red[BPD_NW] = v;
  }
  __syncthreads();
  const int am = static_cast<int>(key_v(red[BPD_NW]));
  if constexpr (RANK) *rank = redc[BPD_NW];
  __syncthreads();
  return am;
}

template <typename T, bool VECTOR, bool RANK>
__global__ void __launch_bounds__(BPD_NT) bpd_verify_kernel(const void* logits, const int32_t* proposals, int k,
                                                           int V, int eos, BpdCrit crit, int32_t* khat_out,
                                                           int32_t* next_out) {
  constexpr int VEC = VECTOR ? Vec16<T>::N : 1;
  __shared__ u64 red[BPD_NW + 1];
  __shared__ int redc[BPD_NW + 1];
  __shared__ u64 part[KMAX];
  __shared__ int am_p[KMAX];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nvec = V / VEC;
  const int64_t row_bytes = static_cast<int64_t>(V) * Elem<T>::BYTES;
  const char* base = reinterpret_cast<const char*>(logits) + static_cast<int64_t>(b) * k * k * row_bytes;
  auto row_ptr = [&](int p, int h) { return base + (static_cast<int64_t>(p) * k + h) * row_bytes; };
  const int32_t* props = proposals + static_cast<int64_t>(b) * k;

  // verify: head 0 at position p must pass proposal p+1
  int n = 1, last_p = -1;
  for (int p = 0; p < k - 1; ++p) {
    const int prop = __ldg(props + p + 1);
    int rank = 0;
    const float xp = RANK ? token_value<T>(row_ptr(p, 0), prop, V) : 0.f;
    const int am = cta_row_argmax<T, VECTOR, RANK>(row_ptr(p, 0), nvec, red, redc, xp, prop, &rank);
    if (tid == 0) am_p[p] = am;
    last_p = p;
    if (!bpd_passes(crit, prop, am, rank, V)) break;
    ++n;
  }
  n = max(n, min(crit.min_accept, k));                 // the minimum block (§5.3), then the EOS cut
  if (eos >= 0) {
    for (int e = 0; e < n; ++e)
      if (__ldg(props + e) == eos) { n = e + 1; break; }
  }
  // accept: the next proposals are every head's argmax at position n-1; head 0
  // there is already known when the checks read that row
  const int p = n - 1;
  const int h0 = (p <= last_p) ? 1 : 0;
  const int nrows = k - h0;
  const int per_row = max(1, BPD_NW / max(1, nrows));
  const int units = nrows * per_row;
  for (int u = warp; u < units; u += BPD_NW) {
    const int r = u / per_row, slice = u - r * per_row;
    const int64_t lo = nvec * slice / per_row, hi = nvec * (slice + 1) / per_row;
    u64 kk = thread_row_best<T, VECTOR>(row_ptr(p, h0 + r), lo + lane, hi, 32);
    kk = warp_max_u64(kk);
    if (lane == 0) part[u] = kk;
  }
  __syncthreads();
  if (tid < nrows) {
    u64 best = 0;
    for (int s2 = 0; s2 < per_row; ++s2) best = part[tid * per_row + s2] > best ? part[tid * per_row + s2] : best;
    next_out[static_cast<int64_t>(b) * k + h0 + tid] = static_cast<int32_t>(key_v(best));
  }
  if (tid == 0) {
    khat_out[b] = n;
    if (h0) next_out[static_cast<int64_t>(b) * k] = am_p[p];
  }
}

// ---------------------------------------------------------------------------------------
// the row argmax of one CTA (BPD_RT threads): each thread tracks the best vector of its
// strided share with packed maxima (ties keep the earlier vector), then the first element
// of that vector equal to its maximum; one reduction over (value, lower index)
// ---------------------------------------------------------------------------------------

constexpr int BPD_RT = 256;
constexpr int BPD_BUF = 64 * 1024;        // shared staging of one row chunk (bulk copy)

// The CTA's staging buffer, its pieces' mbarriers and their phases (bit p: piece p), and
// the row maxima of the single-barrier reduction (two slots, alternating by row).
constexpr int BPD_PIECES = 1;                      // a chunk arrives in this many bulk copies (more measured slower)
struct RowStage {
  unsigned char* buf;
  u64* bar;                                        // [BPD_PIECES]
  u32 phase;
  u64* best;                                       // [2]
  u32 row;                                         // rows scanned so far (selects the slot)
};

__device__ __forceinline__ u32 gt_bf16x2(u32 a, u32 b) {
  u32 d;
  asm("set.gt.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ u32 eq_bf16x2(u32 a, u32 b) {
  u32 d;
  asm("set.eq.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The row's argmax; with RANK also *rank = the number of elements that beat proposal
// `prop` (a larger logit, or an equal one at a lower id).  bf16 vectors count with packed
// compares (each true half of the mask is 16 set bits); an equal element sends the vector
// through the per-element test.
template <typename T, bool VECTOR, bool RANK = false>
__device__ int row_argmax(const char* row, int V, RowStage& st, u64* red, int* status, int* redc = nullptr,
                          int prop = -1, int* rank = nullptr) {
  constexpr int VEC = VECTOR ? Vec16<T>::N : 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  u64 best = 0;
  int cnt = 0;
  float xp = 0.f;
  if constexpr (VECTOR) {
    // the row in chunks of at most BPD_BUF bytes: one bulk copy each, then a scan of the
    // staged vectors from shared memory
    const int nvec = V / VEC;
    constexpr int CH = BPD_BUF / 16;
    float bv = -INFINITY;
    int bi = -1;
    uint4 bq = make_uint4(0, 0, 0, 0);
    for (int c0 = 0; c0 < nvec; c0 += CH) {
      const int nv = min(CH, nvec - c0);
      __syncthreads();                             // the buffer's previous contents are consumed
      if (tid == 0) {
        if (c0 == 0 && !RANK) st.best[(st.row + 1) & 1] = 0ull;   // the next row's slot (read before this barrier)
        for (int pc = 0; pc < BPD_PIECES; ++pc) {
          const int lo = nv * pc / BPD_PIECES, hi = nv * (pc + 1) / BPD_PIECES;
          if (hi == lo) continue;
          mbar_expect_tx(&st.bar[pc], static_cast<u32>(hi - lo) * 16u);
          bulk_g2s(st.buf + lo * 16, row + static_cast<int64_t>(c0 + lo) * 16, static_cast<u32>(hi - lo) * 16u,
                   &st.bar[pc]);
        }
      }
      if (RANK && c0 == 0) xp = token_value<T>(row, prop, V);   // in flight with the copy
      const uint4* v = reinterpret_cast<const uint4*>(st.buf);
      for (int pc = 0; pc < BPD_PIECES; ++pc) {
        const int lo = nv * pc / BPD_PIECES, hi = nv * (pc + 1) / BPD_PIECES;
        if (hi == lo) continue;
        // each piece is scanned as soon as it lands, while the later ones are still in flight
        if (!mbar_wait(&st.bar[pc], (st.phase >> pc) & 1u)) set_status(status, VBS_ETIMEOUT);
        st.phase ^= 1u << pc;
        for (int i = lo + tid; i < hi; i += BPD_RT) {
          const uint4 q = v[i];
          const float m = VecMax<T>::finish(VecMax<T>::fold(q, VecMax<T>::NEG));
          if (m > bv || bi < 0) { bv = m; bi = c0 + i; bq = q; }
          if constexpr (RANK) {
            const int v0 = (c0 + i) * VEC;
            bool tie = true;
            if constexpr (Elem<T>::BYTES == 2) {
              const u32 xb = __float_as_uint(xp) >> 16, refw = xb | (xb << 16);
              cnt += static_cast<int>((__popc(gt_bf16x2(q.x, refw)) + __popc(gt_bf16x2(q.y, refw)) +
                                       __popc(gt_bf16x2(q.z, refw)) + __popc(gt_bf16x2(q.w, refw))) >> 4);
              tie = (eq_bf16x2(q.x, refw) | eq_bf16x2(q.y, refw) | eq_bf16x2(q.z, refw) | eq_bf16x2(q.w, refw)) != 0u;
            }
            if (tie) {
              float x[VEC];
              Vec16<T>::unpack(q, x);
#pragma unroll
              for (int e2 = 0; e2 < VEC; ++e2) {
                if constexpr (Elem<T>::BYTES == 2) cnt += (x[e2] == xp && v0 + e2 < prop) ? 1 : 0;
                else cnt += beats(x[e2], v0 + e2, xp, prop);
              }
            }
          }
        }
      }
    }
    if (bi >= 0) {
      float x[VEC];
      Vec16<T>::unpack(bq, x);
      int e = VEC - 1;
#pragma unroll
      for (int e2 = VEC - 1; e2 >= 0; --e2) e = x[e2] == bv ? e2 : e;
      best = make_key(bv, static_cast<u32>(bi * VEC + e));
    }
  } else {
    if constexpr (RANK) xp = token_value<T>(row, prop, V);
    for (int i = tid; i < V; i += BPD_RT) {
      const float x = Elem<T>::load(row, i);
      const u64 k = make_key(x, static_cast<u32>(i));
      best = k > best ? k : best;
      if constexpr (RANK) cnt += beats(x, i, xp, prop);
    }
  }
  best = warp_max_u64(best);
  if constexpr (!RANK) {
    if (VECTOR) {
      // one barrier: the warps' maxima meet in this row's slot, which thread 0 cleared before
      // the previous row's first barrier
      u64* slot = &st.best[st.row & 1];
      if (lane == 0) atomicMax(slot, best);
      __syncthreads();
      const u64 v = *reinterpret_cast<volatile u64*>(slot);
      st.row += 1;
      return static_cast<int>(key_v(v));
    }
  }
  if constexpr (RANK) cnt = __reduce_add_sync(FULL, cnt);
  if (lane == 0) {
    red[warp] = best;
    if constexpr (RANK) redc[warp] = cnt;
  }
  __syncthreads();
  if (warp == 0) {
    u64 v = lane < BPD_RT / 32 ? red[lane] : 0ull;
    v = warp_max_u64(v);
    if constexpr (RANK) {
      const int cc = __reduce_add_sync(FULL, lane < BPD_RT / 32 ? redc[lane] : 0);
      if (lane == 0) redc[BPD_RT / 32] = cc;
    }
    if (lane == 0) red[BPD_RT / 32] = v;
  }
  __syncthreads();
  if constexpr (RANK) *rank = redc[BPD_RT / 32];
  return static_cast<int>(key_v(red[BPD_RT / 32]));
}

// ---------------------------------------------------------------------------------------
// verify + accept as a persistent work queue
// ---------------------------------------------------------------------------------------
//
// Two kinds of work.  Chains: batch element b's verify (head 0 at positions 0, 1, ...
// while the proposals agree, then head 0 at position khat-1 if the chain did not read
// it), handed out in order by one counter.  Rows: head h at position khat_b - 1, h =
// 1..k-1, which a finished chain publishes into a ready list (it reserves k-1 slots and
// writes each as one 64-bit entry tagged with the call's epoch).  A CTA takes chains
// while any are left, then claims ready slots in order and waits (bounded) until its
// slot is published; every slot is reserved by a chain that is already running, so no
// wait can block the work it waits for.  Only the rows the definition needs are read.
// The counters and the ready list are static device memory, reset by each call's last
// CTA (calls on one stream run one after the other).

constexpr int BPD_MAX_B = 16384;
constexpr int BPD_MAX_READY = BPD_MAX_B * (KMAX - 1);
__device__ unsigned long long g_bpd_ready[BPD_MAX_READY];   // (epoch + 1) << 32 | b << 5 | h
__device__ unsigned g_bpd_epoch;
__device__ int g_bpd_next_chain;
__device__ int g_bpd_ready_head;
__device__ int g_bpd_ready_tail;
__device__ int g_bpd_exited;

__device__ __forceinline__ u64 ld_acquire_u64(const u64* p) {
  u64 v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(u64* p, u64 v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void prefetch_row_l2(const char* p, int64_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(static_cast<unsigned>(bytes)) : "memory");
}

template <typename T, bool VECTOR, bool RANK>
__global__ void __launch_bounds__(BPD_RT, 3) bpd_verify_queue_kernel(const void* logits, const int32_t* proposals, int B,
                                                                  int k, int V, int eos, BpdCrit crit,
                                                                  int32_t* khat_out, int32_t* next_out, int* status) {
  extern __shared__ __align__(128) unsigned char bpd_smem[];
  __shared__ u64 red[BPD_RT / 32 + 1];
  __shared__ int redc[BPD_RT / 32 + 1];
  __shared__ __align__(8) u64 bar[BPD_PIECES];
  __shared__ __align__(8) u64 best2[2];
  __shared__ int s_unit, s_b, s_h, s_q;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int pc = 0; pc < BPD_PIECES; ++pc) mbar_init(&bar[pc], 1);
    fence_mbar_init();
    best2[0] = 0ull;
    best2[1] = 0ull;
  }
  __syncthreads();
  // launched as a programmatic dependent: the set-up above overlaps the previous kernel in
  // the stream; every global access (the queue's counters included) comes after it has
  // completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  RowStage st{bpd_smem, bar, 0u, best2, 0u};
  u64 tag = 0;                                     // this call's ready-list tag, read when first needed
  const int64_t row_bytes = static_cast<int64_t>(V) * Elem<T>::BYTES;
  const int n_rows = B * (k - 1);
  // chains: CTA i starts with chain i, the rest are handed out by the counter (offset by the
  // grid); each CTA asks for its next chain while it runs the current one
  int next_b = static_cast<int>(blockIdx.x);
  for (;;) {
    if (tid == 0) s_unit = next_b;
    __syncthreads();
    const int b = s_unit;
    __syncthreads();
    if (b >= B) break;
    if (tid == 0) next_b = static_cast<int>(gridDim.x) + atomicAdd(&g_bpd_next_chain, 1);
    if (!VBS_CHECK(b >= 0, 21, b, status)) break;
    const char* base = reinterpret_cast<const char*>(logits) + static_cast<int64_t>(b) * k * k * row_bytes;
    const int32_t* props = proposals + static_cast<int64_t>(b) * k;
    int checks = k - 1;                            // proposals up to an EOS need no checks past it
    if (eos >= 0)
      for (int e = 0; e < k; ++e)
        if (__ldg(props + e) == eos) { checks = min(checks, e); break; }
    int n = 1, am = -1, last = -1;
    for (int p = 0; p < checks; ++p) {
      const char* row = base + static_cast<int64_t>(p) * k * row_bytes;
      const int prop = __ldg(props + p + 1);
      int rank = 0;
      if constexpr (RANK) {
        am = row_argmax<T, VECTOR, true>(row, V, st, red, status, redc, prop, &rank);
      } else {
        am = row_argmax<T, VECTOR>(row, V, st, red, status);
      }
      last = p;
      if (!bpd_passes(crit, prop, am, rank, V)) break;
      ++n;
    }
    // the minimum block (§5.3), then the EOS cut: proposals past an EOS are not accepted
    if (crit.min_accept > n) {
      n = min(crit.min_accept, k);
      if (eos >= 0)
        for (int e = 0; e < n; ++e)
          if (__ldg(props + e) == eos) { n = e + 1; break; }
    }
    if (last != n - 1)                             // khat - 1 not read by the checks: head 0 there
      am = row_argmax<T, VECTOR>(base + static_cast<int64_t>(n - 1) * k * row_bytes, V, st, red, status);
    if (tid == 0) {
      khat_out[b] = n;
      next_out[static_cast<int64_t>(b) * k] = am;
      if (k > 1) {
        if (!tag) tag = static_cast<u64>(*reinterpret_cast<volatile unsigned*>(&g_bpd_epoch) + 1u) << 32;
        const int slot = atomicAdd(&g_bpd_ready_tail, k - 1);
        for (int h = 1; h < k; ++h)
          if (VBS_CHECK(slot + h - 1 < BPD_MAX_READY, 20, slot + h - 1, status))
            st_release_u64(&g_bpd_ready[slot + h - 1], tag | (static_cast<u64>(b) << 5) | static_cast<u64>(h));
      }
    }
  }
  // published rows: head h at position khat_b - 1
  if (tid == 0 && !tag) tag = static_cast<u64>(*reinterpret_cast<volatile unsigned*>(&g_bpd_epoch) + 1u) << 32;
  for (;;) {
    if (tid == 0) {
      const int r = atomicAdd(&g_bpd_ready_head, 1);
      s_unit = r;
      if (r < n_rows && VBS_CHECK(r < BPD_MAX_READY, 22, r, status)) {
        u64 e = 0;
        u32 it = 0;
        while (((e = ld_acquire_u64(&g_bpd_ready[r])) >> 32) != (tag >> 32)) {
          if (++it > (1u << 24)) { set_status(status, VBS_ETIMEOUT); break; }
          __nanosleep(32);
        }
        const int b = static_cast<int>((e & 0xffffffffull) >> 5);
        s_b = min(b, B - 1);
        s_h = max(1, min(static_cast<int>(e & 31u), k - 1));
        s_q = max(1, min(*reinterpret_cast<volatile int32_t*>(khat_out + s_b), k)) - 1;
      }
    }
    __syncthreads();
    const int r = s_unit, b = s_b, h = s_h, q = s_q;
    __syncthreads();
    if (r >= n_rows) break;
    const char* row = reinterpret_cast<const char*>(logits) + ((static_cast<int64_t>(b) * k + q) * k + h) * row_bytes;
    const int am = row_argmax<T, VECTOR>(row, V, st, red, status);
    if (tid == 0) next_out[static_cast<int64_t>(b) * k + h] = am;
  }
  // the last CTA out resets the queue and moves the ready list to the next epoch (the next
  // call on the stream touches them only after its griddepcontrol.wait, i.e. once this grid
  // has completed)
  if (tid == 0) {
    if (atomicAdd(&g_bpd_exited, 1) == static_cast<int>(gridDim.x) - 1) {
      g_bpd_next_chain = 0;
      g_bpd_ready_head = 0;
      g_bpd_ready_tail = 0;
      g_bpd_exited = 0;
      __threadfence();
      atomicAdd(&g_bpd_epoch, 1u);
    }
  }
}

template <typename T, bool VECTOR>
__global__ void __launch_bounds__(256) bpd_propose_kernel(const void* logits, int V, int32_t* proposals) {
  constexpr int VEC = VECTOR ? Vec16<T>::N : 1;
  __shared__ u64 red[9];
  const int64_t row_bytes = static_cast<int64_t>(V) * Elem<T>::BYTES;
  const char* row = reinterpret_cast<const char*>(logits) + blockIdx.x * row_bytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  u64 k = thread_row_best<T, VECTOR>(row, tid, V / VEC, 256);
  k = warp_max_u64(k);
  if (lane == 0) red[warp] = k;
  __syncthreads();
  if (warp == 0) {
    u64 v = lane < 8 ? red[lane] : 0ull;
    v = warp_max_u64(v);
    if (lane == 0) proposals[blockIdx.x] = static_cast<int32_t>(key_v(v));
  }
}

int launch_bpd_propose(const void* logits, int B, int k, int V, int dtype, bool vec_ok, int32_t* proposals,
                       cudaStream_t s) {
  const int grid = B * k;
  if (grid == 0) return VBS_OK;
  if (dtype == VBS_BF16) {
    if (vec_ok) bpd_propose_kernel<bf16_t, true><<<grid, 256, 0, s>>>(logits, V, proposals);
    else bpd_propose_kernel<bf16_t, false><<<grid, 256, 0, s>>>(logits, V, proposals);
  } else {
    if (vec_ok) bpd_propose_kernel<float, true><<<grid, 256, 0, s>>>(logits, V, proposals);
    else bpd_propose_kernel<float, false><<<grid, 256, 0, s>>>(logits, V, proposals);
  }
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

template <typename T, bool VECTOR, bool RANK>
static int launch_queue(int grid, const void* logits, const int32_t* proposals, int B, int k, int V, int eos,
                        const BpdCrit& crit, int32_t* khat, int32_t* next, int* status, cudaStream_t s) {
  const int smem = VECTOR ? BPD_BUF : 0;
  static std::atomic<unsigned long long> attr_done{0};   // one per kernel instantiation
  if (VECTOR && !smem_attr_once(bpd_verify_queue_kernel<T, VECTOR, RANK>, BPD_BUF, attr_done)) return VBS_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(BPD_RT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bpd_verify_queue_kernel<T, VECTOR, RANK>, logits, proposals, B, k, V, eos, crit,
                            khat, next, status) == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

template <typename T, bool VECTOR>
static int launch_verify(const void* logits, const int32_t* proposals, int B, int k, int V, int eos,
                         const BpdCrit& crit, int32_t* khat, int32_t* next, int* status, int num_sms, cudaStream_t s) {
  const bool rank = crit.mode == VBS_BPD_TOPK;
  if (B <= BPD_MAX_B) {
    const int grid = std::min(B * k, num_sms * 3);  // three CTAs (three staged rows) per SM
    return rank ? launch_queue<T, VECTOR, true>(grid, logits, proposals, B, k, V, eos, crit, khat, next, status, s)
                : launch_queue<T, VECTOR, false>(grid, logits, proposals, B, k, V, eos, crit, khat, next, status, s);
  }
  if (rank) bpd_verify_kernel<T, VECTOR, true><<<B, BPD_NT, 0, s>>>(logits, proposals, k, V, eos, crit, khat, next);
  else bpd_verify_kernel<T, VECTOR, false><<<B, BPD_NT, 0, s>>>(logits, proposals, k, V, eos, crit, khat, next);
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

int launch_bpd_verify(const void* logits, const int32_t* proposals, int B, int k, int V, int dtype, bool vec_ok,
                      int eos, const BpdCrit& crit, int32_t* khat, int32_t* next, int* status, int num_sms,
                      cudaStream_t s) {
  if (B == 0) return VBS_OK;
  if (dtype == VBS_BF16)
    return vec_ok ? launch_verify<bf16_t, true>(logits, proposals, B, k, V, eos, crit, khat, next, status, num_sms, s)
                  : launch_verify<bf16_t, false>(logits, proposals, B, k, V, eos, crit, khat, next, status, num_sms, s);
  return vec_ok ? launch_verify<float, true>(logits, proposals, B, k, V, eos, crit, khat, next, status, num_sms, s)
                : launch_verify<float, false>(logits, proposals, B, k, V, eos, crit, khat, next, status, num_sms, s);
}

unsigned long long bpd_check_record() { return read_check_record(); }

}  // namespace vbs
