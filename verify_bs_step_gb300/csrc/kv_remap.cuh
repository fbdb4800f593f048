// The paged KV remap of one sentence, run by one CTA of NT threads: shared by the
// standalone remap kernel and the beam-step kernel that fuses it after its merge.
//
// What is computed follows "9.2 贪心搜索与束搜索：确定性与近似搜索" §9.2.2 (the
// cache paragraph: row r continues from the cache of its parent beam_idx[r]; a
// paged cache rewrites block-table entries and copies only when a shared block is
// written).  The remap is sentence-local (blocks are never shared across
// sentences): the sentence's table rows, reference counts and free stack are
// loaded into shared memory in one round, new references are counted before old
// ones are dropped (a block shared by parent and child never reaches zero in
// between), freed blocks return to the stack in ascending id order, one warp makes
// the block holding position t_valid exclusive to every live row (a fresh block, or
// a copy-on-write task when it is shared; blocks and tasks go to the rows in row
// order), and the sentence's tasks go to its own slots of the task list.
#pragma once

#include "common.cuh"
#include "bs_internal.h"

namespace vbs {

struct RemapShared {
  int nold[WMAX], par[WMAX], nnew[WMAX], tail[WMAX];
  int top;
};

// Shared-memory ints the remap needs besides RemapShared.
__host__ __device__ inline int64_t remap_scratch_ints(const PagedArgs& a) {
  return static_cast<int64_t>(a.W) * a.MB + 3 * static_cast<int64_t>(a.S);
}

// Every thread of the CTA calls it (it synchronises the CTA three times); bi is the
// step's beam_idx (global rows, -1 for a finished sentence's pads).  The sentence's
// copy-on-write tasks go to its own task slots [b*W, (b+1)*W), unused slots get 0
// filled positions, so no two sentences contend and the copy kernel needs no count.
template <int NT>
__device__ void paged_remap_sentence(const PagedArgs& a, int b, const int32_t* bi, int t_valid, int32_t* rs,
                                     RemapShared& sh) {
  const int W = a.W, S = a.S, MB = a.MB;
  const int r0 = b * W;
  int32_t* old = rs;                   // [W][MB]
  int32_t* rc = old + W * MB;          // [S] counts now
  int32_t* rc0 = rc + S;               // [S] counts before
  int32_t* stk = rc0 + S;              // [S]
  const int tid = threadIdx.x;

  // one round of loads: everything the sentence's remap reads (a finished sentence's
  // state is read and left as it is); each of the first W threads checks its row's parent
  // every load is issued before the first one is used: registers first, then shared memory
  constexpr int LU = 4;                                   // entries per thread per round
  const int nt = W * MB;
  const int32_t* tab = a.table + static_cast<int64_t>(r0) * MB;
  const int32_t* rcg = a.refcnt + static_cast<int64_t>(b) * S;
  const int32_t* stg = a.stack + static_cast<int64_t>(b) * S;
  int live = 0;
  int nold = 0, p = -1, top = 0;
  if (tid < W) {
    nold = a.nblk[r0 + tid];
    p = __ldcg(bi + r0 + tid);                            // a fused caller wrote it in this kernel
  }
  if (tid == 0) top = a.top[b];
  for (int i0 = 0; i0 < nt || i0 < S; i0 += NT * LU) {
    int tv[LU], rv[LU], sv[LU];
#pragma unroll
    for (int u = 0; u < LU; ++u) {
      const int i = i0 + u * NT + tid;
      tv[u] = i < nt ? tab[i] : 0;
      rv[u] = i < S ? rcg[i] : 0;
      sv[u] = i < S ? stg[i] : 0;
    }
#pragma unroll
    for (int u = 0; u < LU; ++u) {
      const int i = i0 + u * NT + tid;
      if (i < nt) old[i] = tv[u];
      if (i < S) {
        rc[i] = rv[u];
        rc0[i] = rv[u];
        stk[i] = sv[u];
      }
    }
  }
  if (tid < W) {
    sh.nold[tid] = nold;
    if (p >= 0) {
      live = 1;
      if (p < r0 || p >= r0 + W) {
        set_status(a.status, VBS_EINVAL);
        p = -1;
      }
    }
    sh.par[tid] = p;
  }
  if (tid == 0) sh.top = top;
  if (!__syncthreads_or(live)) {                          // a finished sentence: nothing moves
    if (tid < W) a.tasks[r0 + tid] = make_int4(0, 0, 0, 0);
    return;
  }

  // reference counts after the step: +1 for every entry a row takes from its parent, -1
  // for every entry it drops (the final counts do not depend on the order)
  for (int i = tid; i < W * MB; i += NT) {
    const int w = i / MB, s = i - w * MB;
    const int p = sh.par[w];
    if (p < 0) continue;
    if (s < sh.nold[p - r0]) {
      const int blk = old[(p - r0) * MB + s] - b * S;
      if (blk >= 0 && blk < S) atomicAdd(&rc[blk], 1);
      else set_status(a.status, VBS_EINVAL);
    }
    if (s < sh.nold[w]) {
      const int blk = old[w * MB + s] - b * S;
      if (blk >= 0 && blk < S) atomicSub(&rc[blk], 1);
    }
  }
  __syncthreads();
  if (tid < 32) {
    // one warp: freed blocks go back on the stack in ascending id order, then the rows'
    // tail blocks are decided in parallel (lane w for row w) with the outcome of taking the
    // rows one after the other in row order
    const int lane = tid;
    int top = sh.top;
    for (int j0 = 0; j0 < S; j0 += 32) {
      const int j = j0 + lane;
      const bool freed = j < S && rc0[j] > 0 && rc[j] == 0;
      const u32 m = __ballot_sync(FULL, freed);
      const int pos = top + __popc(m & ((1u << lane) - 1u));
      if (freed && pos < S) stk[pos] = b * S + j;
      top = min(S, top + __popc(m));
    }
    __syncwarp();
    // the block holding position t_valid must be exclusive to each live row: a row whose
    // parent ends just before it takes a fresh block (kind 1); a row whose parent's block
    // there is shared keeps it if it is the lowest such row, else copies it (kind 2)
    const int i = t_valid / a.block, fill = t_valid % a.block;
    const u32 lt = (1u << lane) - 1u;
    int kind = 0, blk = -1, nnew = 0;
    if (lane < W) {
      const int p = sh.par[lane];
      if (p < 0) {
        nnew = sh.nold[lane];
      } else {
        const int n = sh.nold[p - r0];
        nnew = n;
        if (n == i) {
          kind = 1;
        } else if (n == i + 1) {
          blk = old[(p - r0) * MB + i];
          if (blk < b * S || blk >= (b + 1) * S) set_status(a.status, VBS_EINVAL);
          else if (rc[blk - b * S] != 1) kind = 2;
        } else {
          set_status(a.status, VBS_EINVAL);               // the table does not match t_valid
        }
      }
    }
    bool keeper = kind == 2;
    for (int q = 0; q < W; ++q) {                         // a lower row copying the same block
      const int qk = __shfl_sync(FULL, kind, q), qb = __shfl_sync(FULL, blk, q);
      if (q < lane && qk == 2 && qb == blk) keeper = false;
    }
    if (keeper) kind = 0;
    // fresh blocks come off the stack in row order; rows past the stack's end get none
    const u32 need = __ballot_sync(FULL, kind != 0);
    const int idx = __popc(need & lt);
    int tail = -1;
    if (kind != 0) {
      const int nb = idx < top ? stk[top - 1 - idx] : -1;
      if (idx < top && (nb < b * S || nb >= (b + 1) * S)) {
        set_status(a.status, VBS_EINVAL);                 // a corrupt free stack
        kind = 0;
      } else if (idx < top) {
        tail = nb;
        rc[tail - b * S] = 1;
        if (kind == 1) nnew = i + 1;
        else atomicSub(&rc[blk - b * S], 1);
      } else {
        set_status(a.status, VBS_ENOMEM);
        kind = 0;
      }
    }
    const u32 cow = __ballot_sync(FULL, kind == 2);
    const int n_tasks = __popc(cow);
    if (kind == 2) a.tasks[r0 + __popc(cow & lt)] = make_int4(blk, tail, fill, 0);
    if (lane >= n_tasks && lane < W) a.tasks[r0 + lane] = make_int4(0, 0, 0, 0);
    if (lane < W) {
      sh.tail[lane] = tail;
      sh.nnew[lane] = nnew;
    }
    if (lane == 0) {
      sh.top = top - min(__popc(need), top);
      if (n_tasks) atomicAdd(a.cow_slots, static_cast<unsigned long long>(n_tasks) * fill * (a.L * 2 * a.H));
    }
  }
  __syncthreads();

  // write back
  const int ti = t_valid / a.block;
  for (int i = tid; i < W * MB; i += NT) {
    const int w = i / MB, s = i - w * MB;
    const int p = sh.par[w];
    if (p < 0) continue;
    int v = s < sh.nold[p - r0] ? old[(p - r0) * MB + s] : -1;
    if (s == ti && sh.tail[w] >= 0) v = sh.tail[w];
    if (s < sh.nnew[w]) a.table[static_cast<int64_t>(r0 + w) * MB + s] = v;
  }
  if (tid < W) a.nblk[r0 + tid] = sh.nnew[tid];
  for (int j = tid; j < S; j += NT) {
    a.refcnt[static_cast<int64_t>(b) * S + j] = rc[j];
    a.stack[static_cast<int64_t>(b) * S + j] = stk[j];
  }
  if (tid == 0) a.top[b] = sh.top;
}

}  // namespace vbs
