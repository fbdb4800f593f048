// KV-cache reorder by beam_idx (sm_103a): naive gather and paged block table
// with copy-on-write.
//
// What is computed follows "9.2 贪心搜索与束搜索：确定性与近似搜索" §9.2.2 (the
// cache paragraph: row r continues from the cache of its parent beam_idx[r]; the
// naive way gathers every layer's K and V; a paged cache rewrites block-table
// entries and copies only when a shared block is written) and §9.2.4 (prompt
// sharing).
//
// The naive gather moves long contiguous runs, so it runs on the bulk-copy (TMA)
// engine: one elected thread per CTA keeps a ring of shared-memory stages full
// with cp.async.bulk global->shared loads (completing on mbarriers) and drains
// them with cp.async.bulk shared->global stores (bulk groups).  The paged
// copy-on-write moves short scattered runs, warp per run with 16-byte vectors.
// The remap of the paged table is sentence-local (blocks are never shared
// across sentences), so it runs one CTA per sentence on shared-memory copies of
// the sentence's table rows, reference counts and free stack, with a
// deterministic allocation order; each sentence writes its copy-on-write tasks
// to its own task slots (kv_remap.cuh).  Both paged kernels are programmatic
// dependents of their predecessor in the stream.

#include "common.cuh"
#include "bs_internal.h"
#include "kv_remap.cuh"

namespace vbs {

constexpr int KV_STAGES = 6;
constexpr int KV_CHUNK = 16384;       // bytes per bulk copy
constexpr int KV_CTAS_PER_SM = 2;

// ---------------------------------------------------------------------------------------
// the bulk-copy engine: items i = blockIdx.x, blockIdx.x + gridDim.x, ...;
// Map(i, &src, &dst, &bytes) returns false (or bytes == 0) for an item with nothing to copy.
// ---------------------------------------------------------------------------------------

template <class Map>
__device__ void bulk_copy_items(const Map& map, int64_t n_items, int* status) {
  extern __shared__ __align__(128) unsigned char kv_smem[];
  __shared__ __align__(8) u64 bars[KV_STAGES];
  if (threadIdx.x != 0) return;
  for (int s = 0; s < KV_STAGES; ++s) mbar_init(&bars[s], 1);
  fence_mbar_init();

  const int64_t first = blockIdx.x, step = gridDim.x;
  const int64_t n_mine = first < n_items ? (n_items - first + step - 1) / step : 0;
  auto issue_load = [&](int64_t k) {
    const int st = static_cast<int>(k % KV_STAGES);
    const char* src = nullptr;
    char* dst = nullptr;
    u32 bytes = 0;
    map(first + k * step, src, dst, bytes);
    mbar_expect_tx(&bars[st], bytes);
    if (bytes) bulk_g2s(kv_smem + st * KV_CHUNK, src, bytes, &bars[st]);
  };
  for (int64_t k = 0; k < KV_STAGES - 1 && k < n_mine; ++k) issue_load(k);
  bool ok = true;
  for (int64_t k = 0; k < n_mine; ++k) {
    const int st = static_cast<int>(k % KV_STAGES);
    if (ok && !mbar_wait(&bars[st], static_cast<u32>((k / KV_STAGES) & 1))) {
      set_status(status, VBS_ETIMEOUT);
      ok = false;
    }
    const char* src = nullptr;
    char* dst = nullptr;
    u32 bytes = 0;
    map(first + k * step, src, dst, bytes);
    if (ok && bytes) bulk_s2g(dst, kv_smem + st * KV_CHUNK, bytes);
    bulk_commit();
    if (k + KV_STAGES - 1 < n_mine) {
      bulk_wait_read<1>();                 // the stage of item k-1 is free again
      if (ok) issue_load(k + KV_STAGES - 1);
    }
  }
  bulk_wait<0>();
  if (!ok) {
    // give loads still in flight a bounded chance to land before the CTA exits
    for (int s = 0; s < KV_STAGES; ++s) mbar_wait(&bars[s], 0, 1u << 16);
  }
}

// ---------------------------------------------------------------------------------------
// naive gather: dst[l, kv, r, h, 0:t] = src[l, kv, beam_idx[r], h, 0:t]
// ---------------------------------------------------------------------------------------

struct NaiveMap {
  const char* src;
  char* dst;
  const int32_t* bi;
  int H, rows;
  int64_t seg_stride, copy_bytes, nch;
  int* status;
  __device__ void operator()(int64_t item, const char*& s, char*& d, u32& bytes) const {
    const int64_t c = item % nch;
    const int64_t seg = item / nch;
    const int h = static_cast<int>(seg % H);
    const int r = static_cast<int>((seg / H) % rows);
    const int64_t lkv = seg / (static_cast<int64_t>(H) * rows);
    const int p = __ldg(bi + r);
    bytes = 0;
    if (p < 0) return;
    if (p >= rows) {                                  // not a row of the cache: nothing is copied
      set_status(status, VBS_EINPUT);
      return;
    }
    const int64_t off = c * KV_CHUNK;
    const int64_t rem = copy_bytes - off;
    bytes = static_cast<u32>(rem < KV_CHUNK ? rem : KV_CHUNK);
    s = src + ((lkv * rows + p) * H + h) * seg_stride + off;
    d = dst + ((lkv * rows + r) * H + h) * seg_stride + off;
  }
};

__global__ void __launch_bounds__(32) kv_naive_bulk_kernel(NaiveMap map, int64_t n_items, int* status) {
  bulk_copy_items(map, n_items, status);
}

// Element-wise fallback for layouts the bulk engine cannot take (alignment).
template <typename W>
__global__ void kv_naive_plain_kernel(const char* src, char* dst, const int32_t* bi, int H, int rows,
                                      int64_t seg_stride, int64_t copy_words, int64_t n_segs, int* status) {
  const int64_t total = n_segs * copy_words;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t seg = i / copy_words, w = i % copy_words;
    const int h = static_cast<int>(seg % H);
    const int r = static_cast<int>((seg / H) % rows);
    const int64_t lkv = seg / (static_cast<int64_t>(H) * rows);
    const int p = __ldg(bi + r);
    if (p < 0) continue;
    if (p >= rows) {                                  // not a row of the cache: nothing is copied
      set_status(status, VBS_EINPUT);
      continue;
    }
    const W* s = reinterpret_cast<const W*>(src + ((lkv * rows + p) * H + h) * seg_stride);
    W* d = reinterpret_cast<W*>(dst + ((lkv * rows + r) * H + h) * seg_stride);
    d[w] = s[w];
  }
}

int launch_kv_naive(const KvGeom& g, const void* src, void* dst, const int32_t* beam_idx, bool bulk_ok,
                    int elem_bytes, int* status, int num_sms, cudaStream_t s) {
  const int64_t n_segs = static_cast<int64_t>(g.L) * 2 * g.rows * g.H;
  if (g.copy_bytes == 0 || n_segs == 0) return VBS_OK;
  if (bulk_ok) {
    NaiveMap m{static_cast<const char*>(src), static_cast<char*>(dst), beam_idx, g.H, g.rows,
               g.seg_stride, g.copy_bytes, (g.copy_bytes + KV_CHUNK - 1) / KV_CHUNK, status};
    const int64_t n_items = n_segs * m.nch;
    const size_t smem = static_cast<size_t>(KV_STAGES) * KV_CHUNK;
    static std::atomic<unsigned long long> attr_done{0};
    if (!smem_attr_once(kv_naive_bulk_kernel, static_cast<int>(smem), attr_done)) return VBS_ECUDA;
    const int grid = static_cast<int>(std::min<int64_t>(n_items, static_cast<int64_t>(num_sms) * KV_CTAS_PER_SM));
    kv_naive_bulk_kernel<<<grid, 32, smem, s>>>(m, n_items, status);
  } else {
    const int64_t grid = std::min<int64_t>(static_cast<int64_t>(num_sms) * 8, 1 << 16);
    const char* sp = static_cast<const char*>(src);
    char* dp = static_cast<char*>(dst);
    if (g.copy_bytes % 4 == 0 && g.seg_stride % 4 == 0 && elem_bytes % 4 == 0)
      kv_naive_plain_kernel<uint32_t><<<static_cast<int>(grid), 256, 0, s>>>(
          sp, dp, beam_idx, g.H, g.rows, g.seg_stride, g.copy_bytes / 4, n_segs, status);
    else if (g.copy_bytes % 2 == 0 && g.seg_stride % 2 == 0)
      kv_naive_plain_kernel<uint16_t><<<static_cast<int>(grid), 256, 0, s>>>(
          sp, dp, beam_idx, g.H, g.rows, g.seg_stride, g.copy_bytes / 2, n_segs, status);
    else
      kv_naive_plain_kernel<uint8_t><<<static_cast<int>(grid), 256, 0, s>>>(
          sp, dp, beam_idx, g.H, g.rows, g.seg_stride, g.copy_bytes, n_segs, status);
  }
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

// ---------------------------------------------------------------------------------------
// paged: remap + reference counts + free stack + copy-on-write tasks (one CTA per sentence)
// ---------------------------------------------------------------------------------------

constexpr int REMAP_NT = 256;

// Launch with programmatic stream serialization: the kernel may be scheduled while its
// predecessor in the stream finishes; it calls griddepcontrol.wait before touching memory.
template <typename... KArgs, typename... Args>
static int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

__global__ void __launch_bounds__(REMAP_NT) kv_paged_remap_kernel(const PagedArgs a, const int32_t* bi,
                                                                  int t_valid) {
  extern __shared__ int32_t rs[];
  __shared__ RemapShared sh;
  // launched as a programmatic dependent of the beam step: wait for it (and everything
  // before it) before the first global access
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  paged_remap_sentence<REMAP_NT>(a, blockIdx.x, bi, t_valid, rs, sh);
}

int launch_kv_paged_remap(const PagedArgs& a, const int32_t* beam_idx, int t_valid, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(remap_scratch_ints(a)) * sizeof(int32_t);
  if (smem > 200 * 1024) return VBS_EINVAL;
  static std::atomic<int> attr[64];                // the limit set so far, per device
  if (!smem_attr_at_least(kv_paged_remap_kernel, static_cast<int>(smem), attr)) return VBS_ECUDA;
  return launch_pdl(kv_paged_remap_kernel, dim3(a.B), dim3(REMAP_NT), smem, s, a, beam_idx, t_valid);
}

// copy-on-write: task q copies the filled slots of every (l, kv, h) run of a block
struct CowMap {
  const char* pool;
  const int4* tasks;
  int task_cap;
  int n_runs;                       // L * 2 * H
  int64_t block_bytes, run_bytes, slot_bytes;
  int64_t n_blocks;                 // blocks in the pool
  int* status;
  __device__ void operator()(int64_t item, const char*& s, char*& d, u32& bytes) const {
    const int q = static_cast<int>(item / n_runs);
    const int run = static_cast<int>(item % n_runs);
    const int4 t = tasks[q];
    bytes = static_cast<u32>(t.z * slot_bytes);
    if (bytes && !VBS_CHECK(t.x >= 0 && t.x < n_blocks && t.y >= 0 && t.y < n_blocks, 11, t.x, status)) bytes = 0;
    s = pool + t.x * block_bytes + run * run_bytes;
    d = const_cast<char*>(pool) + t.y * block_bytes + run * run_bytes;
  }
};

// Copy-on-write items are short (one run's filled slots, a few KB) and scattered, so
// the copy is warp-per-item with plain 16-byte vectors: each lane issues up to COW_U loads
// before its stores, and 32 warps per SM keep about 128 KB in flight, which is what HBM
// latency needs at full bandwidth.  Items cover every row's task slot; a slot the remap
// left empty (0 filled positions) copies nothing.
constexpr int COW_NT = 256;
constexpr int COW_CTAS_PER_SM = 4;
constexpr int COW_U = 8;

__device__ __forceinline__ void st_stream16(void* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(COW_NT) kv_cow_vec_kernel(CowMap map) {
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the remap's tasks
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t n_items = static_cast<int64_t>(map.task_cap) * map.n_runs;
  const int lane = threadIdx.x & 31;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * (COW_NT / 32);
  for (int64_t item = static_cast<int64_t>(blockIdx.x) * (COW_NT / 32) + (threadIdx.x >> 5); item < n_items;
       item += nw) {
    const char* src;
    char* dst;
    u32 bytes;
    map(item, src, dst, bytes);
    const int nv = static_cast<int>(bytes / 16);
    for (int base = 0; base < nv; base += 32 * COW_U) {
      uint4 v[COW_U];
#pragma unroll
      for (int u = 0; u < COW_U; ++u) {
        const int i = base + u * 32 + lane;
        if (i < nv) v[u] = ld_stream16(src + static_cast<int64_t>(i) * 16);
      }
#pragma unroll
      for (int u = 0; u < COW_U; ++u) {
        const int i = base + u * 32 + lane;
        if (i < nv) st_stream16(dst + static_cast<int64_t>(i) * 16, v[u]);
      }
    }
  }
}

__global__ void kv_cow_plain_kernel(CowMap map) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t n_items = static_cast<int64_t>(map.task_cap) * map.n_runs;
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const char* s;
    char* d;
    u32 bytes;
    map(item, s, d, bytes);
    for (u32 i = threadIdx.x; i < bytes; i += blockDim.x) d[i] = s[i];
  }
}

int launch_kv_paged_cow(const PagedArgs& a, bool bulk_ok, int num_sms, cudaStream_t s) {
  const int n_runs = a.L * 2 * a.H;
  const int64_t run_bytes = static_cast<int64_t>(a.block) * a.slot_bytes;
  CowMap m{a.pool, a.tasks, a.task_cap, n_runs, a.block_bytes, run_bytes, a.slot_bytes,
           static_cast<int64_t>(a.B) * a.S, a.status};
  if (bulk_ok) return launch_pdl(kv_cow_vec_kernel, dim3(num_sms * COW_CTAS_PER_SM), dim3(COW_NT), 0, s, m);
  return launch_pdl(kv_cow_plain_kernel, dim3(num_sms * KV_CTAS_PER_SM), dim3(256), 0, s, m);
}

unsigned long long kv_check_record() { return read_check_record(); }

}  // namespace vbs
