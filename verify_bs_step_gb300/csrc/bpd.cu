// Blockwise parallel decoding: predict (per-head argmax) and verify + accept
// (sm_103a).
//
// What is computed follows "Blockwise Parallel Decoding for Deep Autoregressive
// Models" (papercache notes), §3 (predict, verify: the largest khat such that
// every proposal up to khat equals the base model's argmax given the proposals
// before it; khat >= 1; accept) and §4 (the combined scoring and proposal model:
// the verify call also yields the next iteration's proposals from position
// khat).  Layout: logits[b, p, h, :] is head h+1 at proposal position p+1.
//
// One CTA per batch element.  The verify checks are sequential (each decides
// whether the next row is needed), so only the rows the definition needs are
// read: head 0 at positions 0..khat-1 (at most k-1 of them), then the k heads
// at position khat-1, the already-known head 0 reused.  Argmax ties go to the
// lower token id, through a (logit, token) key where a larger key is better.

#include "common.cuh"
#include "bs_internal.h"

namespace vbs {

constexpr int BPD_NT = 512;
constexpr int BPD_NW = BPD_NT / 32;
constexpr int BPD_U = 8;

// Best key of the vectors [i0, i1) of one row, for this thread (strided by `stride`).
template <typename T, bool VECTOR>
__device__ __forceinline__ u64 thread_row_best(const char* row, int64_t i0, int64_t i1, int64_t stride) {
  constexpr int VEC = VECTOR ? Vec16<T>::N : 1;
  u64 best = 0;
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
        }
      }
    }
  }
  return best;
}

template <typename T, bool VECTOR>
__device__ __forceinline__ int cta_row_argmax(const char* row, int64_t nvec, u64* red) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  u64 k = thread_row_best<T, VECTOR>(row, tid, nvec, BPD_NT);
  k = warp_max_u64(k);
  if (lane == 0) red[warp] = k;
  __syncthreads();
  if (warp == 0) {
    u64 v = lane < BPD_NW ? red[lane] : 0ull;
    v = warp_max_u64(v);
    if (lane == 0) red[BPD_NW] = v;
  }
  __syncthreads();
  const int am = static_cast<int>(key_v(red[BPD_NW]));
  __syncthreads();
  return am;
}

template <typename T, bool VECTOR>
__global__ void __launch_bounds__(BPD_NT) bpd_verify_kernel(const void* logits, const int32_t* proposals, int k,
                                                           int V, int eos, int32_t* khat_out, int32_t* next_out) {
  constexpr int VEC = VECTOR ? Vec16<T>::N : 1;
  __shared__ u64 red[BPD_NW + 1];
  __shared__ u64 part[KMAX];
  __shared__ int am_p[KMAX];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nvec = V / VEC;
  const int64_t row_bytes = static_cast<int64_t>(V) * Elem<T>::BYTES;
  const char* base = reinterpret_cast<const char*>(logits) + static_cast<int64_t>(b) * k * k * row_bytes;
  auto row_ptr = [&](int p, int h) { return base + (static_cast<int64_t>(p) * k + h) * row_bytes; };
  const int32_t* props = proposals + static_cast<int64_t>(b) * k;

  // verify: head 0 at position p must reproduce proposal p+1
  int n = 1, last_p = -1;
  for (int p = 0; p < k - 1; ++p) {
    const int am = cta_row_argmax<T, VECTOR>(row_ptr(p, 0), nvec, red);
    if (tid == 0) am_p[p] = am;
    last_p = p;
    if (__ldg(props + p + 1) != am) break;
    ++n;
  }
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

int launch_bpd_verify(const void* logits, const int32_t* proposals, int B, int k, int V, int dtype, bool vec_ok,
                      int eos, int32_t* khat, int32_t* next, cudaStream_t s) {
  if (B == 0) return VBS_OK;
  if (dtype == VBS_BF16) {
    if (vec_ok) bpd_verify_kernel<bf16_t, true><<<B, BPD_NT, 0, s>>>(logits, proposals, k, V, eos, khat, next);
    else bpd_verify_kernel<bf16_t, false><<<B, BPD_NT, 0, s>>>(logits, proposals, k, V, eos, khat, next);
  } else {
    if (vec_ok) bpd_verify_kernel<float, true><<<B, BPD_NT, 0, s>>>(logits, proposals, k, V, eos, khat, next);
    else bpd_verify_kernel<float, false><<<B, BPD_NT, 0, s>>>(logits, proposals, k, V, eos, khat, next);
  }
  return cudaGetLastError() == cudaSuccess ? VBS_OK : VBS_ECUDA;
}

}  // namespace vbs
