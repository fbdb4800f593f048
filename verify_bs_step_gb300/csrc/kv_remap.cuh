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
// between), freed blocks return to the stack in ascending id order, thread 0 makes
// the block holding position t_valid exclusive to every live row in row order (a
// fresh block, or a copy-on-write task when it is shared), and the sentence's
// tasks go to its own slots of the task list.
#pragma once

#include "common.cuh"
#include "bs_internal.h"

namespace vbs {

struct RemapShared {
  int nold[WMAX], par[WMAX], nnew[WMAX], tail[WMAX], kept[WMAX];
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
    // freed blocks go back on the stack in ascending id order
    for (int j0 = 0; j0 < S; j0 += 32) {
      const int j = j0 + tid;
      const bool freed = j < S && rc0[j] > 0 && rc[j] == 0;
      const u32 m = __ballot_sync(FULL, freed);
      const int pos = sh.top + __popc(m & ((1u << tid) - 1u));
      if (freed && pos < S) stk[pos] = b * S + j;
      __syncwarp();
      if (tid == 0) sh.top = min(S, sh.top + __popc(m));
      __syncwarp();
    }
    // make the block holding position t_valid exclusive to each live row, in row order
    if (tid == 0) {
      const int i = t_valid / a.block, fill = t_valid % a.block;
      int n_kept = 0, n_tasks = 0;
      for (int w = 0; w < W; ++w) {
        sh.tail[w] = -1;
        const int p = sh.par[w];
        if (p < 0) { sh.nnew[w] = sh.nold[w]; continue; }
        const int n = sh.nold[p - r0];
        sh.nnew[w] = n;
        if (n == i) {                                     // a fresh block, nothing to copy
          if (sh.top == 0) { set_status(a.status, VBS_ENOMEM); continue; }
          const int nb = stk[--sh.top];
          rc[nb - b * S] = 1;
          sh.tail[w] = nb;
          sh.nnew[w] = i + 1;
        } else if (n == i + 1) {
          const int blk = old[(p - r0) * MB + i];
          if (rc[blk - b * S] == 1) continue;
          bool is_kept = false;
          for (int q = 0; q < n_kept; ++q) is_kept |= sh.kept[q] == blk;
          if (!is_kept) { sh.kept[n_kept++] = blk; continue; }   // the lowest row keeps the shared block
          if (sh.top == 0) { set_status(a.status, VBS_ENOMEM); continue; }
          const int nb = stk[--sh.top];
          rc[nb - b * S] = 1;
          rc[blk - b * S] -= 1;
          sh.tail[w] = nb;
          a.tasks[r0 + n_tasks++] = make_int4(blk, nb, fill, 0);
        } else {
          set_status(a.status, VBS_EINVAL);               // the table does not match t_valid
        }
      }
      for (int q = n_tasks; q < W; ++q) a.tasks[r0 + q] = make_int4(0, 0, 0, 0);
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
