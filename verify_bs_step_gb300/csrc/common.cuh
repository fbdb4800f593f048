// Device helpers shared by the libvbs kernels (sm_103a).
#pragma once

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "vbs.h"

namespace vbs {

using u32 = uint32_t;
using u64 = unsigned long long;

constexpr u32 FULL = 0xffffffffu;
constexpr float LOG2E_F = 1.4426950408889634f;
constexpr double LN2_D = 0.69314718055994530942;

// ------------------------------------------------------------------------------------
// element access
// ------------------------------------------------------------------------------------

// bf16 -> fp32 is exact: the 16 bits are the top half of the fp32 pattern.
__device__ __forceinline__ float bf16_lo(u32 w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(u32 w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int BYTES = 4;
  __device__ __forceinline__ static float load(const void* p, int64_t i) {
    return __ldg(reinterpret_cast<const float*>(p) + i);
  }
};
struct bf16_t { uint16_t bits; };
template <> struct Elem<bf16_t> {
  static constexpr int BYTES = 2;
  __device__ __forceinline__ static float load(const void* p, int64_t i) {
    u32 h = __ldg(reinterpret_cast<const unsigned short*>(p) + i);
    return __uint_as_float(h << 16);
  }
};

// Streaming 16-byte load that does not allocate in L1 (each logit is read once).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Prefetch [p, p + bytes) into L2, one 128-byte line per call, lines i = lane, lane + nl, ...
__device__ __forceinline__ void prefetch_l2(const void* p, int64_t bytes, int lane, int nl) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(p) & ~static_cast<uintptr_t>(127);
  const uintptr_t a1 = reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(bytes);
  for (uintptr_t q = a0 + static_cast<uintptr_t>(lane) * 128; q < a1; q += static_cast<uintptr_t>(nl) * 128)
    asm volatile("prefetch.global.L2 [%0];" :: "l"(q));
}

// Unpack one 16-byte vector into VEC floats (8 bf16 or 4 fp32).
template <typename T> struct Vec16;
template <> struct Vec16<bf16_t> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4& q, float (&x)[8]) {
    x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x); x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
    x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z); x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
  }
};
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& q, float (&x)[4]) {
    x[0] = __uint_as_float(q.x); x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z); x[3] = __uint_as_float(q.w);
  }
};

// Elementwise max of two packed bf16 pairs (PTX max.bf16x2).
__device__ __forceinline__ u32 max_bf16x2(u32 a, u32 b) {
  u32 d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The largest value held in one 16-byte vector word set (bf16 or fp32), as fp32.
template <typename T> struct VecMax;
template <> struct VecMax<bf16_t> {
  static constexpr u32 NEG = 0xff80ff80u;           // two bf16 -inf
  __device__ __forceinline__ static u32 fold(const uint4& q, u32 acc) {
    return max_bf16x2(max_bf16x2(acc, max_bf16x2(q.x, q.y)), max_bf16x2(q.z, q.w));
  }
  __device__ __forceinline__ static float finish(u32 acc) { return fmaxf(bf16_lo(acc), bf16_hi(acc)); }
};
template <> struct VecMax<float> {
  static constexpr u32 NEG = 0xff800000u;           // fp32 -inf
  __device__ __forceinline__ static u32 fold(const uint4& q, u32 acc) {
    float m = fmaxf(fmaxf(__uint_as_float(acc), __uint_as_float(q.x)),
                    fmaxf(__uint_as_float(q.y), fmaxf(__uint_as_float(q.z), __uint_as_float(q.w))));
    return __float_as_uint(m);
  }
  __device__ __forceinline__ static float finish(u32 acc) { return __uint_as_float(acc); }
};

// ------------------------------------------------------------------------------------
// arithmetic
// ------------------------------------------------------------------------------------

// 2^a through the SFU (PTX ex2.approx.ftz.f32): ex2(-inf) = 0.
__device__ __forceinline__ float ex2(float a) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}

// ------------------------------------------------------------------------------------
// ordered keys: a larger key is a better (logit, token) pair
// ------------------------------------------------------------------------------------

// Monotone map of fp32 bits to u32 (bigger float -> bigger integer; -0 < +0).
__device__ __forceinline__ u32 ord_f32(float x) {
  u32 b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unord_f32(u32 o) {
  u32 b = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
  return __uint_as_float(b);
}
// key = (logit, then lower token first). 0 is below every real key.
__device__ __forceinline__ u64 make_key(float x, u32 v) {
  return (static_cast<u64>(ord_f32(x)) << 32) | static_cast<u64>(~v);
}
__device__ __forceinline__ float key_x(u64 k) { return unord_f32(static_cast<u32>(k >> 32)); }
__device__ __forceinline__ u32 key_v(u64 k) { return ~static_cast<u32>(k & 0xffffffffull); }

__device__ __forceinline__ u64 shfl64(u64 v, int src) {
  u32 lo = __shfl_sync(FULL, static_cast<u32>(v), src);
  u32 hi = __shfl_sync(FULL, static_cast<u32>(v >> 32), src);
  return (static_cast<u64>(hi) << 32) | lo;
}
__device__ __forceinline__ u64 shfl64_up(u64 v, int d) {
  u32 lo = __shfl_up_sync(FULL, static_cast<u32>(v), d);
  u32 hi = __shfl_up_sync(FULL, static_cast<u32>(v >> 32), d);
  return (static_cast<u64>(hi) << 32) | lo;
}
__device__ __forceinline__ u64 shfl64_xor(u64 v, int m) {
  u32 lo = __shfl_xor_sync(FULL, static_cast<u32>(v), m);
  u32 hi = __shfl_xor_sync(FULL, static_cast<u32>(v >> 32), m);
  return (static_cast<u64>(hi) << 32) | lo;
}
__device__ __forceinline__ u64 warp_max_u64(u64 v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) {
    u64 o = shfl64_xor(v, m);
    v = o > v ? o : v;
  }
  return v;
}

// A warp-resident list of the K best keys (K <= 32): lane i holds the i-th best,
// lanes >= K hold 0.  `thr` is the K-th best (0 while fewer than K are held).
struct WarpTopK {
  u64 item;
  u64 thr;
  float thr_x;     // logit of thr, -inf while the list is not full
  int K;

  __device__ __forceinline__ void reset(int k) {
    K = k; item = 0; thr = 0; thr_x = -INFINITY;
  }
  __device__ __forceinline__ void refresh(int lane) {
    (void)lane;
    thr = shfl64(item, K - 1);
    thr_x = thr ? key_x(thr) : -INFINITY;
  }
  // Insert one warp-uniform key (caller checked key > thr).
  __device__ __forceinline__ void insert(u64 key, int lane) {
    u32 better = __ballot_sync(FULL, lane < K && item > key);
    int pos = __popc(better);
    u64 up = shfl64_up(item, 1);
    if (lane > pos && lane < K) item = up;
    if (lane == pos) item = key;
    refresh(lane);
  }
  // Bitonic sort of one key per lane, descending; keep the first K.
  __device__ __forceinline__ void init_from_lanes(u64 key, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        u64 o = shfl64_xor(key, stride);
        bool lower = (lane & stride) == 0;
        bool desc = (lane & size) == 0;   // final pass (size 32): all descending
        bool take_max = (lower == desc);
        u64 mx = o > key ? o : key, mn = o > key ? key : o;
        key = take_max ? mx : mn;
      }
    }
    item = lane < K ? key : 0ull;
    refresh(lane);
  }
};

// ------------------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA) wrappers
// ------------------------------------------------------------------------------------

__device__ __forceinline__ u32 smem_u32(const void* p) {
  return static_cast<u32>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(u64* bar, u32 count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(u64* bar, u32 bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(u64* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
// Barrier among the first `nthreads` threads of the CTA (named barrier `id`, not 0).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}
// Device-scope atomic add with acquire-release ordering; returns the old value.
__device__ __forceinline__ int atomic_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Bounded wait on phase `parity`; returns false if it gave up.
__device__ __forceinline__ bool mbar_wait(u64* bar, u32 parity, u32 max_iter = 1u << 22) {
  u32 ok = 0;
  for (u32 i = 0; i < max_iter; ++i) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    if (ok) return true;
  }
  return false;
}
// global -> shared bulk copy completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, u32 bytes, u64* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_u32(dst_smem)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// shared -> global bulk copy, tracked by bulk groups.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src_smem, u32 bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               :: "l"(dst), "r"(smem_u32(src_smem)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed groups still read shared memory.
template <int N> __device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory");
}
template <int N> __device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" :: "n"(N) : "memory");
}

__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------------------------
// device bounds checks of the checked build (compiled with VBS_CHECKED)
// ------------------------------------------------------------------------------------
//
// VBS_CHECK(cond, site, index, status) guards one indexed access: in the checked build a
// false condition records (site, index) in this translation unit's record (the first
// failure wins), sets VBS_EBOUNDS in the status word and yields false, so the caller skips
// the access; the normal build compiles it to true.  Sites are numbered per file; the
// record is read by vbs_checked_record().

#ifdef VBS_CHECKED
static __device__ unsigned long long g_check_record;   // ((site + 1) << 40) | index, 0 = none

__device__ __forceinline__ bool check_impl(bool ok, int site, long long index, int* status) {
  if (!ok) {
    const unsigned long long rec = (static_cast<unsigned long long>(site + 1) << 40) |
                                   (static_cast<unsigned long long>(index) & 0xffffffffffull);
    atomicCAS(&g_check_record, 0ull, rec);
    set_status(status, VBS_EBOUNDS);
  }
  return ok;
}
#define VBS_CHECK(cond, site, index, status) \
  ::vbs::check_impl(static_cast<bool>(cond), (site), static_cast<long long>(index), (status))

// Read (then clear) this translation unit's record: 0 if no check failed.
static inline unsigned long long read_check_record() {
  unsigned long long rec = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&rec, g_check_record, sizeof(rec)) != cudaSuccess) return ~0ull;
  cudaMemcpyToSymbol(g_check_record, &zero, sizeof(zero));
  return rec;
}
#else
#define VBS_CHECK(cond, site, index, status) true
static inline unsigned long long read_check_record() { return 0; }
#endif

// Raise a kernel's dynamic shared-memory limit once per device (the attribute is per
// device and function); `done` holds one bit per device already set.
template <typename F>
inline bool smem_attr_once(F* fn, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  const unsigned long long bit = 1ull << dev;
  if (done.load(std::memory_order_acquire) & bit) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  done.fetch_or(bit, std::memory_order_acq_rel);
  return true;
}

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the current device;
// `set` holds the limit already set per device (a kernel whose need varies by call).
template <typename F>
inline bool smem_attr_at_least(F* fn, int bytes, std::atomic<int> (&set)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  int cur = set[dev].load(std::memory_order_acquire);
  if (bytes <= cur || bytes <= 48 * 1024) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  while (cur < bytes && !set[dev].compare_exchange_weak(cur, bytes, std::memory_order_acq_rel)) {
  }
  return true;
}

}  // namespace vbs
