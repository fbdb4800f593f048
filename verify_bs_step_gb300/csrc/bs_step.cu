// Fused batched beam-search step (sm_103a).
//
// One launch per step.  The R = B*W logit rows are cut into G equal ranges of
// the flattened [R, V] index space (G = a whole number of waves over the SMs);
// a CTA streams its range once, keeping per thread an online log-sum-exp and per
// warp a resident list of the K = 2W best (logit, token) pairs, and publishes one
// partial (log2-domain max, scaled sum, K keys) per row segment.  An atomic
// ticket per row makes the last CTA of a row merge its partials (LSE in fp64,
// top-K), and a ticket per sentence makes the last row-merger of a sentence run
// the sentence merge: the W-way merge of the rows' sorted lists into the 2W best
// candidates by (score desc, flat index asc), the walk that moves EOS hits into
// the finished set, the stopping test, the outputs and the in-place sequence
// gather.  No CTA ever waits on another.
//
// What is computed follows "Transformers中的Beam Search高效实现" (section
// 多个样本同时进行beam search: log_softmax, add beam_scores, view [batch, W*V],
// top-k, beam_id = j // V, token_id = j % V, BeamHypotheses.add / is_done, pad
// rows of finished sentences) and "9.2 贪心搜索与束搜索" (§9.2.2 four sub-steps,
// "何时结束" early_stopping modes; §9.2.3 length penalty).

#include <cfloat>
#include <cmath>

#include "common.cuh"
#include "bs_internal.h"

namespace vbs {

constexpr int BS_NT = 512;
constexpr int BS_NW = BS_NT / 32;
constexpr int BS_U = 4;          // 16-byte vectors in flight per thread
constexpr int SEQ_TILE = 256;

__device__ __forceinline__ double lp_dev(double n, double alpha, int kind) {
  if (alpha == 0.0) return 1.0;
  return kind == VBS_LP_GNMT ? pow((5.0 + n) / 6.0, alpha) : pow(n, alpha);
}

__device__ __forceinline__ int64_t first_cta(int64_t r, int64_t V, int64_t per) { return (r * V) / per; }
__device__ __forceinline__ int nparts(int64_t r, int64_t V, int64_t per) {
  return static_cast<int>(((r + 1) * V - 1) / per - (r * V) / per + 1);
}

// Merge (M, l) pairs in the log2 domain: sum = l * 2^M.
__device__ __forceinline__ void lse_merge(float& M, float& l, float M2, float l2) {
  float Mn = fmaxf(M, M2);
  if (Mn == -INFINITY) { M = Mn; l = 0.f; return; }
  l = l * ex2(M - Mn) + l2 * ex2(M2 - Mn);
  M = Mn;
}

// Warp 0 selects the K best of n keys held in shared memory (destroys them).
// Lane i < K returns the i-th best (0 when fewer than i+1 keys exist).
__device__ u64 warp_select_topk(u64* keys, int n, int K, int lane) {
  u64 mine = 0;
  for (int round = 0; round < K; ++round) {
    u64 best = 0;
    int bi = -1;
    for (int c = lane; c < n; c += 32) {
      u64 k = keys[c];
      if (k > best) { best = k; bi = c; }
    }
    u64 g = warp_max_u64(best);
    if (g == 0) break;
    if (bi >= 0 && best == g) keys[bi] = 0;
    if (lane == round) mine = g;
    __syncwarp();
  }
  return mine;
}

struct BsShared {
  u64 keys[BS_NW * KMAX];            // warp lists -> CTA list; later row / sentence lists
  float M[BS_NW], l[BS_NW];
  int flag;
  // sentence merge
  double lse[WMAX];
  float s[WMAX];
  double f_ns[WMAX];
  int f_len[WMAX], f_serial[WMAX], f_src[WMAX];
  int f_count, f_next;
  double f_worst;
  float nb_score[WMAX];
  int nb_tok[WMAX], nb_row[WMAX];
  int done_now;
  int tile[WMAX * SEQ_TILE];
};

// Insert the elements flagged in `cmask` (per lane) into the warp list.
template <int VEC>
__device__ __forceinline__ void insert_pending(WarpTopK& tk, u32 cmask, const float (&x)[VEC], u32 vb,
                                               int lane) {
  u32 pend = __ballot_sync(FULL, cmask != 0);
  while (pend) {
    int src = __ffs(pend) - 1;
    pend &= pend - 1;
    u32 msk = __shfl_sync(FULL, cmask, src);
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      if (msk & (1u << e)) {
        u64 k = shfl64(make_key(x[e], vb + e), src);
        if (k > tk.thr) tk.insert(k, lane);
      }
    }
  }
}

// Stream one row segment [v0, v1): online LSE per thread, top-K per warp; then
// reduce to one partial for the CTA and publish it.
template <typename T, bool VECTOR>
__device__ void stream_segment(const BsArgs& a, BsShared& sh, int r, int64_t v0, int64_t v1, int pidx) {
  constexpr int VEC = VECTOR ? Vec16<T>::N : 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  const int b = r / a.W;
  const bool skip = a.done[b] != 0 || a.scores[r] == -INFINITY;

  float M = -INFINITY, m = -INFINITY, l = 0.f;
  WarpTopK tk;
  tk.reset(K);
  bool inited = false;

  if (!skip) {
    const char* row = reinterpret_cast<const char*>(a.logits) +
                      (static_cast<int64_t>(r) * a.ld + v0) * Elem<T>::BYTES;
    const int64_t n = (v1 - v0) / VEC;
    for (int64_t base = 0; base < n; base += static_cast<int64_t>(BS_NT) * BS_U) {
      uint4 q[BS_U];
      float xs[BS_U];
#pragma unroll
      for (int u = 0; u < BS_U; ++u) {
        int64_t i = base + u * BS_NT + tid;
        if (i < n) {
          if constexpr (VECTOR) q[u] = ld_stream16(row + i * 16);
          else xs[u] = Elem<T>::load(row, i);
        }
      }
#pragma unroll
      for (int u = 0; u < BS_U; ++u) {
        const int64_t i = base + u * BS_NT + tid;
        const bool ok = i < n;
        float x[VEC];
        if constexpr (VECTOR) {
          if (ok) {
            Vec16<T>::unpack(q[u], x);
          } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) x[e] = -INFINITY;
          }
        } else {
          x[0] = ok ? xs[u] : -INFINITY;
        }
        const u32 vb = static_cast<u32>(v0 + i * VEC);
        float vmax = x[0];
#pragma unroll
        for (int e = 1; e < VEC; ++e) vmax = fmaxf(vmax, x[e]);
        // online log-sum-exp in the log2 domain: l = sum 2^(x*log2e - M)
        if (vmax > m) {
          float Mn = vmax * LOG2E_F;
          l *= ex2(M - Mn);
          M = Mn;
          m = vmax;
        }
        if (vmax > -INFINITY) {
          float e2[VEC];
#pragma unroll
          for (int e = 0; e < VEC; ++e) e2[e] = ex2(fmaf(x[e], LOG2E_F, -M));
#pragma unroll
          for (int w = 1; w < VEC; w <<= 1)
#pragma unroll
            for (int e = 0; e + w < VEC; e += 2 * w) e2[e] += e2[e + w];
          l += e2[0];
        }
        // top-K by (logit desc, token asc)
        if (!inited) {
          u64 kmax = 0;
          int emax = -1;
          if (ok) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              u64 k = make_key(x[e], vb + e);
              if (k > kmax) { kmax = k; emax = e; }
            }
          }
          tk.init_from_lanes(kmax, lane);
          u32 cmask = 0;
          if (ok) {
#pragma unroll
            for (int e = 0; e < VEC; ++e)
              if (e != emax && make_key(x[e], vb + e) > tk.thr) cmask |= 1u << e;
          }
          insert_pending<VEC>(tk, cmask, x, vb, lane);
          inited = true;
        } else {
          const bool maybe = ok && vmax >= tk.thr_x;
          if (__any_sync(FULL, maybe)) {
            u32 cmask = 0;
            if (maybe) {
#pragma unroll
              for (int e = 0; e < VEC; ++e)
                if (make_key(x[e], vb + e) > tk.thr) cmask |= 1u << e;
            }
            insert_pending<VEC>(tk, cmask, x, vb, lane);
          }
        }
      }
    }
  }

  // ---- reduce to one partial ----
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float M2 = __shfl_xor_sync(FULL, M, off);
    float l2 = __shfl_xor_sync(FULL, l, off);
    lse_merge(M, l, M2, l2);
  }
  if (lane == 0) { sh.M[warp] = M; sh.l[warp] = l; }
  if (lane < K) sh.keys[warp * K + lane] = inited ? tk.item : 0ull;
  __syncthreads();
  if (warp == 0) {
    float Mw = lane < BS_NW ? sh.M[lane] : -INFINITY;
    float lw = lane < BS_NW ? sh.l[lane] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float M2 = __shfl_xor_sync(FULL, Mw, off);
      float l2 = __shfl_xor_sync(FULL, lw, off);
      lse_merge(Mw, lw, M2, l2);
    }
    u64 top = warp_select_topk(sh.keys, BS_NW * K, K, lane);
    const int64_t slot = static_cast<int64_t>(r) * a.P + pidx;
    if (lane < K) a.part_key[slot * K + lane] = top;
    if (lane == 0) { a.part_M[slot] = Mw; a.part_l[slot] = lw; }
    __threadfence();
  }
  __syncthreads();
}

// Merge row r's partials (CTA-wide; warp 0 does the work).
__device__ void row_merge(const BsArgs& a, BsShared& sh, int r) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int K = a.K;
  const int b = r / a.W;
  const int n = nparts(r, a.V, a.per);
  const int64_t base = static_cast<int64_t>(r) * a.P;
  if (tid < 32) {
    if (a.done[b]) {
      // nothing to merge: the sentence is padded
    } else if (__ldcg(a.scores + r) == -INFINITY) {
      // every candidate of the row is -inf: they rank by token id
      if (lane < K) a.row_key[static_cast<int64_t>(r) * K + lane] =
          lane < a.V ? make_key(-INFINITY, static_cast<u32>(lane)) : 0ull;
      if (lane == 0) a.row_lse[r] = 0.0;
    } else {
      float Mmax = -INFINITY;
      for (int c = lane; c < n; c += 32) Mmax = fmaxf(Mmax, __ldcg(a.part_M + base + c));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) Mmax = fmaxf(Mmax, __shfl_xor_sync(FULL, Mmax, off));
      double acc = 0.0;
      for (int c = lane; c < n; c += 32) {
        float Mc = __ldcg(a.part_M + base + c);
        float lc = __ldcg(a.part_l + base + c);
        if (Mc > -INFINITY) acc += static_cast<double>(lc) * exp2(static_cast<double>(Mc) - Mmax);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(FULL, acc, off);
      for (int c = lane; c < n * K; c += 32) sh.keys[c] = __ldcg(a.part_key + base * K + c);
      __syncwarp();
      u64 top = warp_select_topk(sh.keys, n * K, K, lane);
      if (lane < K) a.row_key[static_cast<int64_t>(r) * K + lane] = top;
      if (lane == 0) {
        double lse = LN2_D * (static_cast<double>(Mmax) + log2(acc));
        if (!(lse < INFINITY)) set_status(a.status, VBS_EINPUT);   // NaN / +inf logits
        a.row_lse[r] = lse;
      }
    }
    __threadfence();
  }
  __syncthreads();
}

// The sentence merge: 2W best candidates, the EOS walk, the stopping test, outputs.
__device__ void sentence_merge(const BsArgs& a, BsShared& sh, int b) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int W = a.W, K = a.K;
  const int r0 = b * W;
  const int t = a.t;
  const int ld = a.seq_ld;
  const bool was_done = a.done[b] != 0;

  if (tid < 32 && !was_done) {
    // load the rows' sorted lists and the finished set
    for (int c = lane; c < W * K; c += 32) sh.keys[c] = __ldcg(a.row_key + static_cast<int64_t>(r0) * K + c);
    if (lane < W) {
      sh.lse[lane] = __ldcg(a.row_lse + r0 + lane);
      sh.s[lane] = __ldcg(a.scores + r0 + lane);
      sh.f_ns[lane] = a.fin_ns[r0 + lane];
      sh.f_len[lane] = a.fin_len[r0 + lane];
      sh.f_serial[lane] = a.fin_serial[r0 + lane];
      sh.f_src[lane] = -1;
    }
    if (lane == 0) {
      sh.f_count = a.fin_count[b];
      sh.f_next = a.fin_next[b];
      sh.f_worst = a.fin_worst[b];
    }
    __syncwarp();
    // W-way merge: lane w walks row w's list
    int h = 0;
    auto cand = [&](int w, int hh, u64& key) -> double {
      key = hh < K ? sh.keys[w * K + hh] : 0ull;
      if (key == 0) return -INFINITY;
      float s = sh.s[w];
      float x = key_x(key);
      if (s == -INFINITY || x == -INFINITY) return -INFINITY;
      return static_cast<double>(s) + static_cast<double>(x) - sh.lse[w];
    };
    int new_cnt = 0;
    double best = 0.0;
    const double lp_t = lp_dev(static_cast<double>(t), a.alpha, a.lp_kind);
    for (int rank = 0; rank < 2 * W && new_cnt < W; ++rank) {
      u64 key;
      double c = lane < W ? cand(lane, h, key) : -INFINITY;
      bool valid = lane < W && key != 0;
      // argmax over lanes by (valid, c desc, row asc)
      double bc = c;
      int bw = valid ? lane : 64;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        double oc = __shfl_xor_sync(FULL, bc, off);
        int ow = __shfl_xor_sync(FULL, bw, off);
        bool take = (ow < 64) && (bw >= 64 || oc > bc || (oc == bc && ow < bw));
        if (take) { bc = oc; bw = ow; }
      }
      if (bw >= 64) break;                       // no candidates left (cannot happen for V >= 2)
      u64 wkey = shfl64(key, bw);
      if (lane == bw) ++h;
      if (lane == 0) {
        if (rank == 0) best = bc;
        const u32 v = key_v(wkey);
        const int parent = r0 + bw;
        if (a.eos >= 0 && static_cast<int>(v) == a.eos) {
          if (rank < W) {
            // BeamHypotheses.add(hyp = parent's sequence, sum = bc), |y| = t
            double ns = bc / lp_t;
            int slot = -1;
            if (sh.f_count < W) {
              slot = sh.f_count++;
              sh.f_worst = fmin(ns, sh.f_worst);
            } else if (ns > sh.f_worst) {
              slot = 0;
              for (int q = 1; q < W; ++q)
                if (sh.f_ns[q] < sh.f_ns[slot] ||
                    (sh.f_ns[q] == sh.f_ns[slot] && sh.f_serial[q] < sh.f_serial[slot]))
                  slot = q;
            }
            if (slot >= 0) {
              sh.f_ns[slot] = ns;
              sh.f_len[slot] = t;
              sh.f_serial[slot] = sh.f_next++;
              sh.f_src[slot] = parent;
              if (sh.f_count >= W && slot >= 0) {
                double wmin = sh.f_ns[0];
                for (int q = 1; q < W; ++q) wmin = fmin(wmin, sh.f_ns[q]);
                sh.f_worst = wmin;
              }
            }
          }
        } else {
          sh.nb_score[new_cnt] = static_cast<float>(bc);
          sh.nb_tok[new_cnt] = static_cast<int>(v);
          sh.nb_row[new_cnt] = parent;
          ++new_cnt;
        }
      }
      new_cnt = __shfl_sync(FULL, new_cnt, 0);
    }
    if (lane == 0) {
      if (new_cnt < W) set_status(a.status, VBS_EINPUT);
      for (int q = new_cnt; q < W; ++q) { sh.nb_score[q] = -INFINITY; sh.nb_tok[q] = a.pad; sh.nb_row[q] = r0; }
      bool done = false;
      if (sh.f_count >= W) {
        if (a.early_stopping == VBS_ES_TRUE) {
          done = true;
        } else {
          double n = (a.early_stopping == VBS_ES_NEVER && a.alpha > 0.0) ? static_cast<double>(a.max_len)
                                                                         : static_cast<double>(t);
          done = sh.f_worst >= best / lp_dev(n, a.alpha, a.lp_kind);
        }
      }
      sh.done_now = done ? 1 : 0;
    }
  }
  if (tid == 0 && was_done) sh.done_now = 1;
  __syncthreads();

  // ---- outputs ----
  if (was_done) {
    if (tid < W) {
      a.beam_idx[r0 + tid] = -1;
      a.tokens[r0 + tid] = a.pad;
      a.scores[r0 + tid] = 0.f;
      a.seqs[static_cast<int64_t>(r0 + tid) * ld + t] = a.pad;
    }
  } else {
    if (tid < W) {
      a.beam_idx[r0 + tid] = sh.nb_row[tid];
      a.tokens[r0 + tid] = sh.nb_tok[tid];
      a.scores[r0 + tid] = sh.nb_score[tid];
      a.fin_ns[r0 + tid] = sh.f_ns[tid];
      a.fin_len[r0 + tid] = sh.f_len[tid];
      a.fin_serial[r0 + tid] = sh.f_serial[tid];
    }
    if (tid == 0) {
      a.fin_count[b] = sh.f_count;
      a.fin_next[b] = sh.f_next;
      a.fin_worst[b] = sh.f_worst;
      a.done[b] = sh.done_now;
    }
    // sequences: gather the parents' columns [0, t) in place, then append the token
    for (int c0 = 0; c0 < t; c0 += SEQ_TILE) {
      const int nc = min(SEQ_TILE, t - c0);
      for (int i = tid; i < W * nc; i += BS_NT) {
        int w = i / nc, c = i - w * nc;
        sh.tile[w * SEQ_TILE + c] = a.seqs[static_cast<int64_t>(r0 + w) * ld + c0 + c];
      }
      __syncthreads();
      for (int i = tid; i < W * nc; i += BS_NT) {
        int w = i / nc, c = i - w * nc;
        a.seqs[static_cast<int64_t>(r0 + w) * ld + c0 + c] = sh.tile[(sh.nb_row[w] - r0) * SEQ_TILE + c];
        if (sh.f_src[w] >= 0)
          a.fin_tok[static_cast<int64_t>(r0 + w) * ld + c0 + c] = sh.tile[(sh.f_src[w] - r0) * SEQ_TILE + c];
      }
      __syncthreads();
    }
    if (tid < W) a.seqs[static_cast<int64_t>(r0 + tid) * ld + t] = sh.nb_tok[tid];
  }
  __threadfence();
  __syncthreads();

  // ---- the last sentence of the step reports all-done ----
  if (tid == 0) {
    int old = atomicAdd(a.glob_ticket, 1);
    sh.flag = old == a.B - 1;
  }
  __syncthreads();
  if (sh.flag) {
    __threadfence();
    int all = 1;
    for (int q = tid; q < a.B; q += BS_NT) all &= __ldcg(a.done + q) != 0;
    all = __syncthreads_and(all);
    if (tid == 0) {
      *a.all_done_dev = all;
      if (a.all_done_out) *a.all_done_out = all;
      *a.glob_ticket = 0;
    }
  }
}

template <typename T, bool VECTOR>
__global__ void __launch_bounds__(BS_NT, 2) bs_step_kernel(const BsArgs a) {
  __shared__ BsShared sh;
  const int64_t total = static_cast<int64_t>(a.R) * a.V;
  const int64_t e0 = static_cast<int64_t>(blockIdx.x) * a.per;
  const int64_t e1 = min(e0 + a.per, total);
  if (e0 >= e1) return;

  // pass 1: stream every row segment of this CTA's range
  for (int64_t e = e0; e < e1;) {
    const int r = static_cast<int>(e / a.V);
    const int64_t v0 = e - static_cast<int64_t>(r) * a.V;
    const int64_t v1 = min(static_cast<int64_t>(a.V), v0 + (e1 - e));
    const int pidx = static_cast<int>(blockIdx.x - first_cta(r, a.V, a.per));
    stream_segment<T, VECTOR>(a, sh, r, v0, v1, pidx);
    e += v1 - v0;
  }
  // pass 2: tickets; the last CTA of a row merges it, the last row of a sentence merges that
  for (int64_t e = e0; e < e1;) {
    const int r = static_cast<int>(e / a.V);
    const int64_t v0 = e - static_cast<int64_t>(r) * a.V;
    const int64_t v1 = min(static_cast<int64_t>(a.V), v0 + (e1 - e));
    e += v1 - v0;
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      int old = atomicAdd(a.row_ticket + r, 1);
      sh.flag = old == nparts(r, a.V, a.per) - 1;
    }
    __syncthreads();
    if (!sh.flag) continue;
    __threadfence();
    row_merge(a, sh, r);
    const int b = r / a.W;
    if (threadIdx.x == 0) {
      a.row_ticket[r] = 0;
      __threadfence();
      int old = atomicAdd(a.sent_ticket + b, 1);
      sh.flag = old == a.W - 1;
    }
    __syncthreads();
    if (!sh.flag) continue;
    __threadfence();
    if (threadIdx.x == 0) a.sent_ticket[b] = 0;
    sentence_merge(a, sh, b);
  }
}

// ---------------------------------------------------------------------------------------
// reset and finalisation
// ---------------------------------------------------------------------------------------

__global__ void bs_reset_kernel(const BsArgs a) {
  const int64_t n = static_cast<int64_t>(a.R) * a.seq_ld;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int c = static_cast<int>(i % a.seq_ld);
    a.seqs[i] = c == 0 ? a.bos : a.pad;
    a.fin_tok[i] = a.pad;
    if (c == 0) {
      int r = static_cast<int>(i / a.seq_ld);
      a.scores[r] = (r % a.W) == 0 ? 0.f : -INFINITY;
      a.fin_ns[r] = 0.0;
      a.fin_len[r] = 0;
      a.fin_serial[r] = 0;
      a.row_ticket[r] = 0;
      if (r < a.B) {
        a.done[r] = 0;
        a.fin_count[r] = 0;
        a.fin_next[r] = 0;
        a.fin_worst[r] = 1e9;
        a.sent_ticket[r] = 0;
      }
      if (r == 0) { *a.glob_ticket = 0; *a.all_done_dev = 0; }
    }
  }
}

// One CTA per sentence: add the live beams of unfinished sentences (|y| = steps
// run), pick the best normalised score (ties: latest list entry), write the row.
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
      const double lpT = lp_dev(static_cast<double>(T), a.alpha, a.lp_kind);
      for (int w = 0; w < W; ++w) {
        double ns = static_cast<double>(scores[r0 + w]) / lpT;
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
            double m = f_ns[0];
            for (int q = 1; q < W; ++q) m = fmin(m, f_ns[q]);
            worst = m;
          }
        }
      }
    }
    int best = 0;
    for (int q = 1; q < count; ++q)
      if (f_ns[q] > f_ns[best] || (f_ns[q] == f_ns[best] && f_serial[q] > f_serial[best])) best = q;
    s_best = best;
    out_score[b] = static_cast<float>(f_ns[best]);
    int n = f_ntok[best];
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

int launch_bs_step(const BsArgs& a, int grid, bool vector_ok, cudaStream_t s) {
  const size_t smem = 0;
  if (a.dtype == VBS_BF16) {
    if (vector_ok) bs_step_kernel<bf16_t, true><<<grid, BS_NT, smem, s>>>(a);
    else bs_step_kernel<bf16_t, false><<<grid, BS_NT, smem, s>>>(a);
  } else {
    if (vector_ok) bs_step_kernel<float, true><<<grid, BS_NT, smem, s>>>(a);
    else bs_step_kernel<float, false><<<grid, BS_NT, smem, s>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

int launch_bs_reset(const BsArgs& a, cudaStream_t s) {
  int64_t n = static_cast<int64_t>(a.R) * a.seq_ld;
  int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096));
  bs_reset_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

int launch_bs_finalize(const BsArgs& a, const float* scores, const int32_t* seqs, int32_t* out_seqs,
                       int32_t* out_len, float* out_score, cudaStream_t s) {
  bs_finalize_kernel<<<a.B, 128, 0, s>>>(a, scores, seqs, out_seqs, out_len, out_score);
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

int bs_threads_per_cta() { return BS_NT; }

}  // namespace vbs
