// In-run memory peaks: the denominators a roofline of this path is read against.
//
// vbs_peak_copy streams src to dst with 16-byte vector loads and stores (read + write
// bytes, like a STREAM copy).  vbs_peak_read only reads: either plain 16-byte vector loads
// (mode 0) or a ring of bulk copies into shared memory with one producer lane and the
// other warps folding a maximum over each stage (mode 1, the access pattern of the beam
// step's streaming loop without its arithmetic).  Each CTA takes one contiguous, equal
// share of the bytes.  Every kernel writes one word per CTA to `sink` so that no load is
// dead code.  Every mbarrier wait is bounded.

#include "common.cuh"

namespace vbs {

namespace {

constexpr int PK_NT = 512;           // threads of the vector-load kernels
constexpr int PK_U = 8;              // 16-byte vectors in flight per thread
constexpr int PR_NC = 512;           // ring kernel: consumer threads
constexpr int PR_STAGE = 32768;      // ring stage bytes
constexpr int PR_NS = 6;             // ring stages

__device__ __forceinline__ u32 fold_max(const uint4& q, u32 acc) {
  return max_bf16x2(max_bf16x2(acc, max_bf16x2(q.x, q.y)), max_bf16x2(q.z, q.w));
}

__global__ void __launch_bounds__(PK_NT) peak_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                          int64_t n16, int64_t per) {
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t b1 = min(b0 + per, n16);
  for (int64_t i = b0 + threadIdx.x; i < b1; i += static_cast<int64_t>(PK_NT) * PK_U) {
    uint4 q[PK_U];
#pragma unroll
    for (int u = 0; u < PK_U; ++u) {
      const int64_t j = i + static_cast<int64_t>(u) * PK_NT;
      if (j < b1) q[u] = ld_stream16(src + j);
    }
#pragma unroll
    for (int u = 0; u < PK_U; ++u) {
      const int64_t j = i + static_cast<int64_t>(u) * PK_NT;
      if (j < b1) dst[j] = q[u];
    }
  }
}

__global__ void __launch_bounds__(PK_NT) peak_read_kernel(const uint4* __restrict__ src, int64_t n16, int64_t per,
                                                          u32* sink) {
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t b1 = min(b0 + per, n16);
  u32 acc = 0xff80ff80u;
  for (int64_t i = b0 + threadIdx.x; i < b1; i += static_cast<int64_t>(PK_NT) * PK_U) {
    uint4 q[PK_U];
#pragma unroll
    for (int u = 0; u < PK_U; ++u) {
      const int64_t j = i + static_cast<int64_t>(u) * PK_NT;
      q[u] = j < b1 ? ld_stream16(src + j) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
    }
#pragma unroll
    for (int u = 0; u < PK_U; ++u) acc = fold_max(q[u], acc);
  }
  for (int o = 16; o > 0; o >>= 1) acc = max_bf16x2(acc, __shfl_xor_sync(FULL, acc, o));
  if ((threadIdx.x & 31) == 0) atomicMax(sink + blockIdx.x, acc);
}

struct RingShared {
  unsigned char ring[PR_NS][PR_STAGE];
  u64 full[PR_NS], empty[PR_NS];
};

// One producer lane fills the ring with bulk copies of at most PR_STAGE bytes; the PR_NC
// consumer threads read each stage once.  The byte range must be 16-byte aligned at both
// ends (the host checks the total; `per` is a multiple of 16).
__global__ void __launch_bounds__(PR_NC + 32, 1) peak_ring_kernel(const char* __restrict__ src, int64_t bytes,
                                                                  int64_t per, u32* sink, int* status) {
  extern __shared__ __align__(128) unsigned char pk_smem[];
  RingShared& sh = *reinterpret_cast<RingShared*>(pk_smem);
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t b1 = min(b0 + per, bytes);
  const int nchunk = b1 > b0 ? static_cast<int>((b1 - b0 + PR_STAGE - 1) / PR_STAGE) : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < PR_NS; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], PR_NC / 32);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == PR_NC / 32) {
    if (lane == 0) {
      for (int c = 0; c < nchunk; ++c) {
        const int s = c % PR_NS;
        if (c >= PR_NS && !mbar_wait(&sh.empty[s], static_cast<u32>(((c / PR_NS) + 1) & 1))) {
          set_status(status, VBS_ETIMEOUT);
        }
        const int64_t off = b0 + static_cast<int64_t>(c) * PR_STAGE;
        const u32 n = static_cast<u32>(min(static_cast<int64_t>(PR_STAGE), b1 - off));
        mbar_expect_tx(&sh.full[s], n);
        bulk_g2s(sh.ring[s], src + off, n, &sh.full[s]);
      }
    }
    return;
  }
  u32 acc = 0xff80ff80u;
  for (int c = 0; c < nchunk; ++c) {
    const int s = c % PR_NS;
    if (!mbar_wait(&sh.full[s], static_cast<u32>((c / PR_NS) & 1))) set_status(status, VBS_ETIMEOUT);
    const int64_t off = b0 + static_cast<int64_t>(c) * PR_STAGE;
    const int n16 = static_cast<int>(min(static_cast<int64_t>(PR_STAGE), b1 - off) / 16);
#pragma unroll
    for (int u = 0; u < PR_STAGE / 16 / PR_NC; ++u) {
      const int i = threadIdx.x + u * PR_NC;
      if (i < n16) acc = fold_max(*reinterpret_cast<const uint4*>(sh.ring[s] + i * 16), acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
  }
  for (int o = 16; o > 0; o >>= 1) acc = max_bf16x2(acc, __shfl_xor_sync(FULL, acc, o));
  if (lane == 0) atomicMax(sink + blockIdx.x, acc);
}

}  // namespace

int launch_peak_copy(const void* src, void* dst, int64_t bytes, int grid, cudaStream_t s) {
  const int64_t n16 = bytes / 16;
  const int64_t per = (n16 + grid - 1) / grid;
  peak_copy_kernel<<<grid, PK_NT, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16, per);
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

int launch_peak_read(const void* src, int64_t bytes, int grid, int mode, u32* sink, int* status, cudaStream_t s) {
  if (mode == 0) {
    const int64_t n16 = bytes / 16;
    const int64_t per = (n16 + grid - 1) / grid;
    peak_read_kernel<<<grid, PK_NT, 0, s>>>(static_cast<const uint4*>(src), n16, per, sink);
    return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
  }
  static std::atomic<unsigned long long> attr_done{0};
  const int smem = static_cast<int>(sizeof(RingShared));
  if (!smem_attr_once(peak_ring_kernel, smem, attr_done)) return VBS_ECUDA;
  const int64_t per = ((bytes + grid - 1) / grid + 15) / 16 * 16;
  peak_ring_kernel<<<grid, PR_NC + 32, smem, s>>>(static_cast<const char*>(src), bytes, per, sink, status);
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

}  // namespace vbs
