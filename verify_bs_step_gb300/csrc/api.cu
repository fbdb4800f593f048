// The C ABI of libvbs: argument checks, context lifetime, workspace layout and
// kernel launches.  No entry point after an init allocates device memory.

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "bs_internal.h"

#define VBS_EXPORT extern "C" __attribute__((visibility("default")))

using vbs::u64;

namespace {

// Status word of the stateless calls (kv_reorder), in static device memory.
__device__ int g_stateless_status;

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// lp(|y|) of "9.2 贪心搜索与束搜索" §9.2.3: GNMT ((5 + |y|) / 6)^alpha or |y|^alpha; alpha = 0 gives 1.
double length_penalty(int n, double alpha, int kind) {
  if (alpha == 0.0) return 1.0;
  return kind == VBS_LP_GNMT ? std::pow((5.0 + n) / 6.0, alpha) : std::pow(static_cast<double>(n), alpha);
}

// One device allocation carved into 256-byte aligned pieces.
struct Carver {
  size_t off = 0;
  char* base = nullptr;
  template <class T> T* take(size_t n) {
    off = (off + 255) & ~static_cast<size_t>(255);
    T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
    off += n * sizeof(T);
    return p;
  }
};

}  // namespace

struct vbs_bs {
  vbs::BsArgs a;
  cudaStream_t stream;
  int step;
  int grid;
  bool reset_done;
  int32_t* seqs_bound;          // the sequence buffer of the current decode
  int32_t* own_seqs;
  void* dev_block;
};

struct vbs_pkv {
  vbs::PagedArgs a;
  cudaStream_t stream;
  int32_t* identity;
  int R;
  void* dev_block;
  char* state;           // table .. top: one contiguous range of the allocation
  char* saved;           // its copy (kv_paged_save / kv_paged_restore)
  size_t state_bytes;
  bool copy_pending;     // bs_step_paged recorded copies that kv_paged_copy has not run
};

VBS_EXPORT const char* vbs_strerror(int status) {
  switch (status) {
    case VBS_OK: return "ok";
    case VBS_EINVAL: return "invalid argument";
    case VBS_ECUDA: return "CUDA error";
    case VBS_ENOMEM: return "out of memory (device allocation or paged block pool)";
    case VBS_ESTATE: return "call does not fit the context's state";
    case VBS_EALIGN: return "misaligned pointer or stride";
    case VBS_ETIMEOUT: return "a bounded device-side wait gave up";
    case VBS_EINPUT: return "input data broke a precondition";
    case VBS_ESCRATCH: return "problem too large for the static scratch of bs_expand_static";
    case VBS_EBOUNDS: return "a device bounds check failed (checked build)";
    default: return "unknown status";
  }
}

VBS_EXPORT int vbs_version(void) { return 100; }

// =====================================================================================
// beam search
// =====================================================================================

VBS_EXPORT int bs_init(vbs_bs** out, int batch, int W, int V, int eos, double alpha, int early_stopping,
                       int lp_kind, int max_len, int bos, int pad, int dtype, vbs_stream_t stream) {
  if (!out) return VBS_EINVAL;
  *out = nullptr;
  if (batch < 1 || batch > 32767 || W < 1 || W > vbs::WMAX || V < 2 || max_len < 1) return VBS_EINVAL;
  if (!(alpha == alpha)) return VBS_EINVAL;
  if (dtype != VBS_F32 && dtype != VBS_BF16) return VBS_EINVAL;
  if (lp_kind != VBS_LP_GNMT && lp_kind != VBS_LP_POWER) return VBS_EINVAL;
  if (early_stopping < VBS_ES_FALSE || early_stopping > VBS_ES_NEVER) return VBS_EINVAL;
  if (eos >= V) return VBS_EINVAL;
  const int64_t R = static_cast<int64_t>(batch) * W;
  if (R * V >= (int64_t{1} << 31) || R * (max_len + 1) >= (int64_t{1} << 31)) return VBS_EINVAL;

  vbs_bs* c = new (std::nothrow) vbs_bs{};
  if (!c) return VBS_ENOMEM;
  vbs::BsArgs& a = c->a;
  a.dtype = dtype;
  a.B = batch;
  a.W = W;
  a.V = V;
  a.K = 2 * W;
  a.R = static_cast<int>(R);
  a.seq_ld = max_len + 1;
  a.eos = eos;
  a.bos = bos;
  a.pad = pad;
  a.early_stopping = early_stopping;
  a.lp_kind = lp_kind;
  a.max_len = max_len;
  a.alpha = alpha;
  c->stream = reinterpret_cast<cudaStream_t>(stream);

  // the flat split: one wave of resident CTAs, ranges of >= 4096 elements,
  // and few enough partials per row for one merge (P * K <= PART_KEYS)
  const int VEC = dtype == VBS_BF16 ? 8 : 4;
  const int64_t total = R * V;
  int64_t G = std::min<int64_t>(static_cast<int64_t>(num_sms()) * vbs::bs_ctas_per_sm(), (total + 4095) / 4096);
  G = std::max<int64_t>(G, 1);
  int64_t per = (total + G - 1) / G;
  const int64_t pmax = vbs::PART_KEYS / a.K - 1;
  per = std::max(per, (V + pmax - 1) / pmax);
  per = (per + VEC - 1) / VEC * VEC;
  G = (total + per - 1) / per;
  a.per = per;
  a.P = static_cast<int>((V + per - 1) / per + 1);
  c->grid = static_cast<int>(G);
  // cluster mode: a cluster of C CTAs per sentence (W / C whole rows each) when the
  // sentence's 2W-best fit one warp's merge and the clusters fit one wave
  a.cluster = 0;
  if (W * a.K <= 32) {
    for (int C = 4; C >= 1; C >>= 1) {
      if (W % C == 0 && W / C <= vbs::BS_NSLOT && static_cast<int64_t>(batch) * C <= num_sms()) {
        a.cluster = C;
        break;
      }
    }
  }

  // vocabulary-shard merges: as many shards per row as the merge kernel's partial buffer holds
  a.shard_max = std::min(vbs::PART_KEYS / a.K, vbs::PART_KEYS / 2 / W);
  Carver cv;
  for (int pass = 0; pass < 2; ++pass) {
    a.shard_M = cv.take<float>(R * a.shard_max);
    a.shard_l = cv.take<float>(R * a.shard_max);
    a.shard_key = cv.take<u64>(R * a.shard_max * a.K);
    a.row_ns = cv.take<int>(R);
    a.part_M = cv.take<float>(R * a.P);
    a.part_l = cv.take<float>(R * a.P);
    a.part_key = cv.take<u64>(R * a.P * a.K);
    a.rtopk_bar = cv.take<unsigned>(R);
    a.row_one = cv.take<int>(R);
    a.row_p0 = cv.take<int>(R);
    a.row_np = cv.take<int>(R);
    a.done_count = cv.take<int>(1);
    a.all_done_dev = cv.take<int32_t>(1);
    a.status = cv.take<int>(1);
    a.done = cv.take<int>(batch);
    a.fin_ns = cv.take<double>(R);
    a.fin_len = cv.take<int>(R);
    a.fin_serial = cv.take<int>(R);
    a.fin_tok = cv.take<int32_t>(R * a.seq_ld);
    a.fin_count = cv.take<int>(batch);
    a.fin_next = cv.take<int>(batch);
    a.fin_worst = cv.take<double>(batch);
    c->own_seqs = cv.take<int32_t>(R * a.seq_ld);
    if (pass == 0) {
      void* p = nullptr;
      if (cudaMalloc(&p, cv.off) != cudaSuccess) {
        cudaGetLastError();
        delete c;
        return VBS_ENOMEM;
      }
      c->dev_block = p;
      cv = Carver{};
      cv.base = static_cast<char*>(p);
    }
  }
  // which CTAs hold each row: row r spans elements [r V, (r + 1) V) of the flat split
  std::vector<int> p0(R), np(R);
  for (int64_t r = 0; r < R; ++r) {
    p0[r] = static_cast<int>((r * V) / per);
    np[r] = static_cast<int>(((r + 1) * V - 1) / per - (r * V) / per + 1);
  }
  bool ok = cudaMemsetAsync(c->dev_block, 0, cv.off, c->stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(a.row_p0, p0.data(), R * sizeof(int), cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(a.row_np, np.data(), R * sizeof(int), cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  const std::vector<int> ones(R, 1);
  ok = ok && cudaMemcpyAsync(a.row_one, ones.data(), R * sizeof(int), cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  ok = ok && cudaStreamSynchronize(c->stream) == cudaSuccess;
  if (!ok) {
    cudaFree(c->dev_block);
    delete c;
    return VBS_ECUDA;
  }
  c->step = 0;
  c->reset_done = false;
  *out = c;
  return VBS_OK;
}

VBS_EXPORT int bs_reset(vbs_bs* c, float* scores, int32_t* seqs) {
  if (!c || !scores) return VBS_EINVAL;
  vbs::BsArgs a = c->a;
  a.scores = scores;
  a.seqs = seqs ? seqs : c->own_seqs;
  int st = vbs::launch_bs_reset(a, c->stream);
  if (st != VBS_OK) return st;
  c->seqs_bound = a.seqs;
  c->step = 0;
  c->reset_done = true;
  return VBS_OK;
}

// The kernel arguments of one step (validated), shared by bs_step and bs_step_paged.
static int step_args(vbs_bs* c, const void* logits, int64_t ld, float* scores, int32_t* seqs, int32_t* beam_idx,
                     int32_t* tokens, int32_t* all_done, vbs::BsArgs& a, bool& vec_ok) {
  if (!c || !logits || !scores || !beam_idx || !tokens) return VBS_EINVAL;
  if (ld < c->a.V) return VBS_EINVAL;
  if (!c->reset_done || c->step >= c->a.max_len) return VBS_ESTATE;
  int32_t* sq = seqs ? seqs : c->own_seqs;
  if (sq != c->seqs_bound) return VBS_ESTATE;
  a = c->a;
  a.logits = logits;
  a.ld = ld;
  a.scores = scores;
  a.seqs = sq;
  a.beam_idx = beam_idx;
  a.tokens = tokens;
  a.all_done_out = all_done;
  a.t = c->step + 1;
  a.lp_t = length_penalty(a.t, a.alpha, a.lp_kind);
  a.lp_bound = (a.early_stopping == VBS_ES_NEVER && a.alpha > 0.0) ? length_penalty(a.max_len, a.alpha, a.lp_kind)
                                                                   : a.lp_t;
  a.lp_tf = static_cast<float>(a.lp_t);
  a.lp_boundf = static_cast<float>(a.lp_bound);
  a.kv_fuse = 0;
  const int es = a.dtype == VBS_BF16 ? 2 : 4;
  const int VEC = 16 / es;
  vec_ok = aligned16(logits) && (ld * es) % 16 == 0 && a.V % VEC == 0;
  return VBS_OK;
}

VBS_EXPORT int bs_step(vbs_bs* c, const void* logits, int64_t ld, float* scores, int32_t* seqs,
                       int32_t* beam_idx, int32_t* tokens, int32_t* all_done) {
  vbs::BsArgs a;
  bool vec_ok = false;
  int st = step_args(c, logits, ld, scores, seqs, beam_idx, tokens, all_done, a, vec_ok);
  if (st != VBS_OK) return st;
  st = vbs::launch_bs_step(a, c->grid, vec_ok, c->stream);
  if (st != VBS_OK) return st;
  c->step += 1;
  return VBS_OK;
}

VBS_EXPORT int bs_step_two_pass(vbs_bs* c, const void* logits, int64_t ld, float* scores, int32_t* seqs,
                                int32_t* beam_idx, int32_t* tokens, int32_t* all_done) {
  vbs::BsArgs a;
  bool vec_ok = false;
  int st = step_args(c, logits, ld, scores, seqs, beam_idx, tokens, all_done, a, vec_ok);
  if (st != VBS_OK) return st;
  st = vbs::launch_bs_step_two_pass(a, vec_ok, c->stream);
  if (st != VBS_OK) return st;
  c->step += 1;
  return VBS_OK;
}

VBS_EXPORT int bs_shard_partial_bytes(vbs_bs* c, int64_t* bytes) {
  if (!c || !bytes) return VBS_EINVAL;
  size_t off_l, off_key, b;
  vbs::shard_partial_layout(c->a.R, c->a.K, &off_l, &off_key, &b);
  *bytes = static_cast<int64_t>(b);
  return VBS_OK;
}

VBS_EXPORT int bs_step_shard(vbs_bs* c, const void* logits_shard, int64_t ld, int v0, int Vs, const float* scores,
                             void* partial) {
  if (!c || !logits_shard || !scores || !partial) return VBS_EINVAL;
  if (v0 < 0 || Vs < 1 || static_cast<int64_t>(v0) + Vs > c->a.V || ld < Vs) return VBS_EINVAL;
  if (!c->reset_done || c->step >= c->a.max_len) return VBS_ESTATE;
  if (!aligned16(partial)) return VBS_EALIGN;
  vbs::BsArgs a = c->a;
  a.logits = logits_shard;
  a.ld = ld;
  a.V = Vs;
  a.vbase = v0;
  a.scores = const_cast<float*>(scores);
  const int es = a.dtype == VBS_BF16 ? 2 : 4;
  const int VEC = 16 / es;
  const bool vec_ok = aligned16(logits_shard) && (ld * es) % 16 == 0 && Vs % VEC == 0;
  return vbs::launch_bs_shard_partial(a, vec_ok, partial, c->stream);
}

VBS_EXPORT int bs_step_merge_shards(vbs_bs* c, int n_shards, const void* partials, float* scores, int32_t* seqs,
                                    int32_t* beam_idx, int32_t* tokens, int32_t* all_done) {
  if (!partials) return VBS_EINVAL;
  vbs::BsArgs a;
  bool vec_ok = false;
  // the logits pointer is unused by the merge: the partials stand in for it
  int st = step_args(c, partials, c ? c->a.V : 0, scores, seqs, beam_idx, tokens, all_done, a, vec_ok);
  if (st != VBS_OK) return st;
  if (n_shards < 1 || n_shards > a.shard_max) return VBS_EINVAL;
  st = vbs::launch_bs_merge_shards(a, n_shards, partials, c->stream);
  if (st != VBS_OK) return st;
  c->step += 1;
  return VBS_OK;
}

VBS_EXPORT int bs_finalize_n(vbs_bs* c, const float* scores, const int32_t* seqs, int n_return, int32_t* out_seqs,
                             int32_t* out_len, float* out_score) {
  if (!c || !scores || !out_seqs || !out_len || !out_score) return VBS_EINVAL;
  if (n_return < 1 || n_return > c->a.W) return VBS_EINVAL;
  if (!c->reset_done) return VBS_ESTATE;
  const int32_t* sq = seqs ? seqs : c->own_seqs;
  if (sq != c->seqs_bound) return VBS_ESTATE;
  vbs::BsArgs a = c->a;
  a.t = c->step;
  a.lp_t = length_penalty(a.t, a.alpha, a.lp_kind);
  return vbs::launch_bs_finalize(a, scores, sq, n_return, out_seqs, out_len, out_score, c->stream);
}

VBS_EXPORT int bs_finalize(vbs_bs* c, const float* scores, const int32_t* seqs, int32_t* out_seqs, int32_t* out_len,
                           float* out_score) {
  return bs_finalize_n(c, scores, seqs, 1, out_seqs, out_len, out_score);
}

VBS_EXPORT int bs_finished(vbs_bs* c, int32_t* count, double* ns, int32_t* len, int32_t* serial, int32_t* tokens,
                           int32_t* done) {
  if (!c) return VBS_EINVAL;
  const vbs::BsArgs& a = c->a;
  const size_t R = static_cast<size_t>(a.R);
  struct Cp { void* dst; const void* src; size_t bytes; } cps[] = {
      {count, a.fin_count, sizeof(int) * a.B},
      {ns, a.fin_ns, sizeof(double) * R},
      {len, a.fin_len, sizeof(int) * R},
      {serial, a.fin_serial, sizeof(int) * R},
      {tokens, a.fin_tok, sizeof(int32_t) * R * a.seq_ld},
      {done, a.done, sizeof(int) * a.B},
  };
  for (const Cp& cp : cps) {
    if (!cp.dst) continue;
    if (cudaMemcpyAsync(cp.dst, cp.src, cp.bytes, cudaMemcpyDeviceToDevice, c->stream) != cudaSuccess)
      return VBS_ECUDA;
  }
  return VBS_OK;
}

VBS_EXPORT int bs_seqs(vbs_bs* c, int32_t** seqs) {
  if (!c || !seqs) return VBS_EINVAL;
  *seqs = c->own_seqs;
  return VBS_OK;
}

VBS_EXPORT int bs_steps(vbs_bs* c, int* steps) {
  if (!c || !steps) return VBS_EINVAL;
  *steps = c->step;
  return VBS_OK;
}

VBS_EXPORT int bs_status(vbs_bs* c) {
  if (!c) return VBS_EINVAL;
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return VBS_ECUDA;
  int h = 0;
  if (cudaMemcpy(&h, c->a.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return VBS_ECUDA;
  if (h != 0) cudaMemset(c->a.status, 0, sizeof(int));
  return h;
}

VBS_EXPORT int bs_destroy(vbs_bs* c) {
  if (!c) return VBS_OK;
  cudaStreamSynchronize(c->stream);
  cudaFree(c->dev_block);
  delete c;
  return VBS_OK;
}

// One expansion step whose scratch is a static device array (no allocation).
VBS_EXPORT int bs_expand_static(const void* logits, int64_t ld, int batch, int W, int V, int dtype,
                                const float* scores_in, float* scores_out, int32_t* beam_idx, int32_t* tokens,
                                vbs_stream_t stream) {
  if (!logits || !scores_in || !scores_out || !beam_idx || !tokens) return VBS_EINVAL;
  if (batch < 1 || W < 1 || W > vbs::WMAX || V < 2 || ld < V) return VBS_EINVAL;
  if (dtype != VBS_F32 && dtype != VBS_BF16) return VBS_EINVAL;
  const int64_t R = static_cast<int64_t>(batch) * W;
  if (R > vbs::STATIC_MAX_ROWS) return VBS_ESCRATCH;
  if (R * V >= (int64_t{1} << 31)) return VBS_EINVAL;
  vbs::BsArgs a{};
  a.logits = logits;
  a.ld = ld;
  a.dtype = dtype;
  a.B = batch;
  a.W = W;
  a.V = V;
  a.K = 2 * W;
  a.R = static_cast<int>(R);
  a.eos = -1;
  a.scores = const_cast<float*>(scores_in);
  a.beam_idx = beam_idx;
  a.tokens = tokens;
  // the same flat split as bs_init
  const int VEC = dtype == VBS_BF16 ? 8 : 4;
  const int64_t total = R * V;
  int64_t G = std::min<int64_t>(static_cast<int64_t>(num_sms()) * vbs::bs_ctas_per_sm(), (total + 4095) / 4096);
  G = std::max<int64_t>(G, 1);
  int64_t per = (total + G - 1) / G;
  const int64_t pmax = vbs::PART_KEYS / a.K - 1;
  per = std::max(per, (V + pmax - 1) / pmax);
  per = (per + VEC - 1) / VEC * VEC;
  G = (total + per - 1) / per;
  a.per = per;
  a.P = static_cast<int>((V + per - 1) / per + 1);
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&a.status), g_stateless_status) != cudaSuccess) return VBS_ECUDA;
  const int es = dtype == VBS_BF16 ? 2 : 4;
  const bool vec_ok = aligned16(logits) && (ld * es) % 16 == 0 && V % VEC == 0;
  return vbs::launch_bs_expand_static(a, static_cast<int>(G), vec_ok, scores_out,
                                      reinterpret_cast<cudaStream_t>(stream));
}

// =====================================================================================
// KV reorder
// =====================================================================================

static bool desc_ok(const vbs_kv_desc* d) {
  return d && d->layers >= 1 && d->heads >= 1 && d->head_dim >= 1 && d->t_max >= 1 &&
         (d->elem_bytes == 1 || d->elem_bytes == 2 || d->elem_bytes == 4 || d->elem_bytes == 8);
}

VBS_EXPORT int kv_reorder(const vbs_kv_desc* d, const void* src, void* dst, const int32_t* beam_idx, int rows,
                          int t_valid, vbs_stream_t stream) {
  if (!desc_ok(d) || !src || !dst || !beam_idx || rows < 1 || t_valid < 0 || t_valid > d->t_max)
    return VBS_EINVAL;
  if (src == dst) return VBS_EINVAL;
  int* status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_stateless_status) != cudaSuccess) return VBS_ECUDA;
  vbs::KvGeom g;
  g.L = d->layers;
  g.H = d->heads;
  g.rows = rows;
  const int64_t slot = static_cast<int64_t>(d->head_dim) * d->elem_bytes;
  g.seg_stride = slot * d->t_max;
  g.copy_bytes = slot * t_valid;
  const bool bulk_ok = slot % 16 == 0 && aligned16(src) && aligned16(dst);
  return vbs::launch_kv_naive(g, src, dst, beam_idx, bulk_ok, d->elem_bytes, status, num_sms(),
                              reinterpret_cast<cudaStream_t>(stream));
}

VBS_EXPORT int vbs_stateless_status(vbs_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return VBS_ECUDA;
  int h = 0;
  if (cudaMemcpyFromSymbol(&h, g_stateless_status, sizeof(int)) != cudaSuccess) return VBS_ECUDA;
  if (h != 0) {
    int z = 0;
    cudaMemcpyToSymbol(g_stateless_status, &z, sizeof(int));
  }
  return h;
}

VBS_EXPORT int kv_paged_init(vbs_pkv** out, const vbs_kv_desc* d, int batch, int W, int S, int block, int MB,
                             void* pool, vbs_stream_t stream) {
  if (!out) return VBS_EINVAL;
  *out = nullptr;
  if (!desc_ok(d) || !pool || batch < 1 || W < 1 || W > vbs::WMAX || S < 1 || block < 1 || MB < 1)
    return VBS_EINVAL;
  if (static_cast<int64_t>(W) * MB + 3 * static_cast<int64_t>(S) > 50000) return VBS_EINVAL;
  vbs_pkv* c = new (std::nothrow) vbs_pkv{};
  if (!c) return VBS_ENOMEM;
  vbs::PagedArgs& a = c->a;
  a.B = batch;
  a.W = W;
  a.S = S;
  a.MB = MB;
  a.block = block;
  a.L = d->layers;
  a.H = d->heads;
  a.slot_bytes = static_cast<int64_t>(d->head_dim) * d->elem_bytes;
  a.block_bytes = static_cast<int64_t>(a.L) * 2 * a.H * block * a.slot_bytes;
  a.pool = static_cast<char*>(pool);
  c->stream = reinterpret_cast<cudaStream_t>(stream);
  const int64_t R = static_cast<int64_t>(batch) * W;
  c->R = static_cast<int>(R);
  const int64_t NB = static_cast<int64_t>(batch) * S;
  Carver cv;
  for (int pass = 0; pass < 2; ++pass) {
    a.table = cv.take<int32_t>(R * MB);
    a.nblk = cv.take<int32_t>(R);
    a.refcnt = cv.take<int32_t>(NB);
    a.stack = cv.take<int32_t>(NB);
    a.top = cv.take<int32_t>(batch);
    const size_t state_end = cv.off;
    c->saved = cv.take<char>(state_end);
    c->state = reinterpret_cast<char*>(a.table);
    c->state_bytes = state_end;
    a.tasks = cv.take<int4>(R);
    a.task_cap = static_cast<int>(R);
    a.cow_slots = cv.take<unsigned long long>(1);
    a.status = cv.take<int>(1);
    c->identity = cv.take<int32_t>(R);
    if (pass == 0) {
      void* p = nullptr;
      if (cudaMalloc(&p, cv.off) != cudaSuccess) {
        cudaGetLastError();
        delete c;
        return VBS_ENOMEM;
      }
      c->dev_block = p;
      cv = Carver{};
      cv.base = static_cast<char*>(p);
    }
  }
  // host image of the initial state: empty tables, full stacks (pops give b*S, b*S+1, ...)
  std::vector<int32_t> table(R * MB, -1), zeros(std::max<int64_t>(R, NB), 0), stack(NB), top(batch, S), ident(R);
  for (int b = 0; b < batch; ++b)
    for (int i = 0; i < S; ++i) stack[static_cast<int64_t>(b) * S + i] = b * S + (S - 1 - i);
  for (int64_t r = 0; r < R; ++r) ident[r] = static_cast<int32_t>(r);
  bool ok = cudaMemsetAsync(c->dev_block, 0, cv.off, c->stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(a.table, table.data(), table.size() * 4, cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(a.stack, stack.data(), stack.size() * 4, cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(a.top, top.data(), top.size() * 4, cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(c->identity, ident.data(), ident.size() * 4, cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  ok = ok && cudaStreamSynchronize(c->stream) == cudaSuccess;
  if (!ok) {
    cudaFree(c->dev_block);
    delete c;
    return VBS_ECUDA;
  }
  *out = c;
  return VBS_OK;
}

static int paged_run(vbs_pkv* c, const int32_t* bi, int t_valid) {
  if (c->copy_pending) return VBS_ESTATE;
  const int64_t need = static_cast<int64_t>(t_valid) / c->a.block + 1;
  if (t_valid < 0 || need > c->a.MB) return VBS_EINVAL;
  int st = vbs::launch_kv_paged_remap(c->a, bi, t_valid, c->stream);
  if (st != VBS_OK) return st;
  const bool bulk_ok = c->a.slot_bytes % 16 == 0 && aligned16(c->a.pool);
  return vbs::launch_kv_paged_cow(c->a, bulk_ok, num_sms(), c->stream);
}

VBS_EXPORT int kv_paged_prefill(vbs_pkv* c, int P) {
  if (!c || P < 0) return VBS_EINVAL;
  const vbs::PagedArgs& a = c->a;
  const int nb = (P + a.block - 1) / a.block;
  if (nb > a.S || nb > a.MB) return VBS_EINVAL;
  const int64_t R = c->R, NB = static_cast<int64_t>(a.B) * a.S;
  std::vector<int32_t> table(R * a.MB, -1), nblk(R, nb), refcnt(NB, 0), stack(NB), top(a.B, a.S - nb);
  for (int b = 0; b < a.B; ++b) {
    for (int i = 0; i < nb; ++i) refcnt[static_cast<int64_t>(b) * a.S + i] = a.W;
    for (int w = 0; w < a.W; ++w)
      for (int i = 0; i < nb; ++i) table[(static_cast<int64_t>(b) * a.W + w) * a.MB + i] = b * a.S + i;
    for (int i = 0; i < a.S; ++i) stack[static_cast<int64_t>(b) * a.S + i] = b * a.S + (a.S - 1 - i);
  }
  bool ok = cudaMemcpyAsync(a.table, table.data(), table.size() * 4, cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(a.nblk, nblk.data(), nblk.size() * 4, cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(a.refcnt, refcnt.data(), refcnt.size() * 4, cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(a.stack, stack.data(), stack.size() * 4, cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(a.top, top.data(), top.size() * 4, cudaMemcpyHostToDevice, c->stream) == cudaSuccess;
  ok = ok && cudaMemsetAsync(a.tasks, 0, sizeof(int4) * c->R, c->stream) == cudaSuccess;
  ok = ok && cudaStreamSynchronize(c->stream) == cudaSuccess;
  c->copy_pending = false;
  return ok ? VBS_OK : VBS_ECUDA;
}

VBS_EXPORT int kv_paged_prepare(vbs_pkv* c, int t_write) {
  if (!c) return VBS_EINVAL;
  return paged_run(c, c->identity, t_write);
}

VBS_EXPORT int kv_paged_reorder(vbs_pkv* c, const int32_t* beam_idx, int t_valid) {
  if (!c || !beam_idx) return VBS_EINVAL;
  return paged_run(c, beam_idx, t_valid);
}

VBS_EXPORT int bs_step_paged(vbs_bs* c, const void* logits, int64_t ld, float* scores, int32_t* seqs,
                             int32_t* beam_idx, int32_t* tokens, int32_t* all_done, vbs_pkv* kv, int t_valid) {
  if (!kv) return VBS_EINVAL;
  vbs::BsArgs a;
  bool vec_ok = false;
  int st = step_args(c, logits, ld, scores, seqs, beam_idx, tokens, all_done, a, vec_ok);
  if (st != VBS_OK) return st;
  if (kv->a.B != a.B || kv->a.W != a.W || kv->stream != c->stream) return VBS_EINVAL;
  if (kv->copy_pending) return VBS_ESTATE;
  const int64_t need = static_cast<int64_t>(t_valid) / kv->a.block + 1;
  if (t_valid < 0 || need > kv->a.MB) return VBS_EINVAL;
  if (vbs::bs_can_fuse_remap(a, kv->a)) {
    a.kv_fuse = 1;
    a.kv_t = t_valid;
    a.kv = kv->a;
    st = vbs::launch_bs_step(a, c->grid, vec_ok, c->stream);
  } else {
    st = vbs::launch_bs_step(a, c->grid, vec_ok, c->stream);
    if (st == VBS_OK) st = vbs::launch_kv_paged_remap(kv->a, beam_idx, t_valid, kv->stream);
  }
  if (st != VBS_OK) return st;
  kv->copy_pending = true;
  c->step += 1;
  return VBS_OK;
}

VBS_EXPORT int kv_paged_copy(vbs_pkv* c) {
  if (!c) return VBS_EINVAL;
  const bool bulk_ok = c->a.slot_bytes % 16 == 0 && aligned16(c->a.pool);
  const int st = vbs::launch_kv_paged_cow(c->a, bulk_ok, num_sms(), c->stream);
  if (st == VBS_OK) c->copy_pending = false;
  return st;
}

VBS_EXPORT int kv_paged_table(vbs_pkv* c, const int32_t** table, int* max_blocks) {
  if (!c || !table || !max_blocks) return VBS_EINVAL;
  *table = c->a.table;
  *max_blocks = c->a.MB;
  return VBS_OK;
}

VBS_EXPORT int kv_paged_counts(vbs_pkv* c, int32_t* refcnt, int32_t* nblk) {
  if (!c) return VBS_EINVAL;
  const size_t NB = static_cast<size_t>(c->a.B) * c->a.S;
  if (refcnt && cudaMemcpyAsync(refcnt, c->a.refcnt, NB * 4, cudaMemcpyDeviceToDevice, c->stream) != cudaSuccess)
    return VBS_ECUDA;
  if (nblk && cudaMemcpyAsync(nblk, c->a.nblk, static_cast<size_t>(c->R) * 4, cudaMemcpyDeviceToDevice,
                              c->stream) != cudaSuccess)
    return VBS_ECUDA;
  return VBS_OK;
}

VBS_EXPORT int kv_paged_save(vbs_pkv* c) {
  if (!c) return VBS_EINVAL;
  return cudaMemcpyAsync(c->saved, c->state, c->state_bytes, cudaMemcpyDeviceToDevice, c->stream) == cudaSuccess
             ? VBS_OK : VBS_ECUDA;
}

VBS_EXPORT int kv_paged_restore(vbs_pkv* c) {
  if (!c) return VBS_EINVAL;
  // copies still pending refer to the state being dropped: forget them
  if (cudaMemsetAsync(c->a.tasks, 0, sizeof(int4) * c->R, c->stream) != cudaSuccess) return VBS_ECUDA;
  c->copy_pending = false;
  return cudaMemcpyAsync(c->state, c->saved, c->state_bytes, cudaMemcpyDeviceToDevice, c->stream) == cudaSuccess
             ? VBS_OK : VBS_ECUDA;
}

VBS_EXPORT int kv_paged_copy_table(vbs_pkv* c, int32_t* out) {
  if (!c || !out) return VBS_EINVAL;
  const size_t n = static_cast<size_t>(c->R) * c->a.MB * 4;
  return cudaMemcpyAsync(out, c->a.table, n, cudaMemcpyDeviceToDevice, c->stream) == cudaSuccess ? VBS_OK
                                                                                                : VBS_ECUDA;
}

VBS_EXPORT int kv_paged_cow_slots(vbs_pkv* c, int64_t* slots) {
  if (!c || !slots) return VBS_EINVAL;
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return VBS_ECUDA;
  unsigned long long h = 0;
  if (cudaMemcpy(&h, c->a.cow_slots, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return VBS_ECUDA;
  *slots = static_cast<int64_t>(h);
  return VBS_OK;
}

VBS_EXPORT int kv_paged_status(vbs_pkv* c) {
  if (!c) return VBS_EINVAL;
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return VBS_ECUDA;
  int h = 0;
  if (cudaMemcpy(&h, c->a.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return VBS_ECUDA;
  if (h != 0) cudaMemset(c->a.status, 0, sizeof(int));
  return h;
}

VBS_EXPORT int kv_paged_destroy(vbs_pkv* c) {
  if (!c) return VBS_OK;
  cudaStreamSynchronize(c->stream);
  cudaFree(c->dev_block);
  delete c;
  return VBS_OK;
}

// =====================================================================================
// blockwise parallel decoding
// =====================================================================================

VBS_EXPORT int bpd_propose(const void* logits, int B, int k, int V, int dtype, int32_t* proposals,
                           vbs_stream_t stream) {
  if (B < 0 || k < 1 || k > vbs::KMAX || V < 1 || (dtype != VBS_F32 && dtype != VBS_BF16)) return VBS_EINVAL;
  if (B > 0 && (!logits || !proposals)) return VBS_EINVAL;
  const int es = dtype == VBS_BF16 ? 2 : 4;
  const bool vec_ok = aligned16(logits) && (static_cast<int64_t>(V) * es) % 16 == 0;
  return vbs::launch_bpd_propose(logits, B, k, V, dtype, vec_ok, proposals, reinterpret_cast<cudaStream_t>(stream));
}

VBS_EXPORT int bpd_verify_approx(const void* logits, const int32_t* proposals, int B, int k, int V, int dtype,
                                 int eos, int criterion, int param, int min_accept, int32_t* khat, int32_t* next,
                                 vbs_stream_t stream) {
  if (B < 0 || k < 1 || k > vbs::KMAX || V < 1 || (dtype != VBS_F32 && dtype != VBS_BF16)) return VBS_EINVAL;
  if (B > 0 && (!logits || !proposals || !khat || !next)) return VBS_EINVAL;
  if (eos >= V) return VBS_EINVAL;
  if (criterion == VBS_BPD_EXACT) param = 0;
  else if (criterion == VBS_BPD_TOPK) { if (param < 1) return VBS_EINVAL; }
  else if (criterion == VBS_BPD_DISTANCE) { if (param < 0) return VBS_EINVAL; }
  else return VBS_EINVAL;
  if (min_accept < 1 || min_accept > k) return VBS_EINVAL;
  const int es = dtype == VBS_BF16 ? 2 : 4;
  const bool vec_ok = aligned16(logits) && (static_cast<int64_t>(V) * es) % 16 == 0;
  int* status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_stateless_status) != cudaSuccess) return VBS_ECUDA;
  const vbs::BpdCrit crit{criterion, param, min_accept};
  return vbs::launch_bpd_verify(logits, proposals, B, k, V, dtype, vec_ok, eos, crit, khat, next, status, num_sms(),
                                reinterpret_cast<cudaStream_t>(stream));
}

VBS_EXPORT int bpd_verify(const void* logits, const int32_t* proposals, int B, int k, int V, int dtype, int eos,
                          int32_t* khat, int32_t* next, vbs_stream_t stream) {
  return bpd_verify_approx(logits, proposals, B, k, V, dtype, eos, VBS_BPD_EXACT, 0, 1, khat, next, stream);
}

// =====================================================================================
// in-run memory peaks
// =====================================================================================

VBS_EXPORT int vbs_peak_copy(const void* src, void* dst, int64_t bytes, int grid, vbs_stream_t stream) {
  if (!src || !dst || bytes <= 0 || grid < 1 || grid > 65535) return VBS_EINVAL;
  if (!aligned16(src) || !aligned16(dst) || bytes % 16 != 0) return VBS_EALIGN;
  return vbs::launch_peak_copy(src, dst, bytes, grid, reinterpret_cast<cudaStream_t>(stream));
}

VBS_EXPORT int vbs_peak_read(const void* src, int64_t bytes, int grid, int mode, uint32_t* sink, vbs_stream_t stream) {
  if (!src || !sink || bytes <= 0 || grid < 1 || grid > 65535 || (mode != 0 && mode != 1)) return VBS_EINVAL;
  if (!aligned16(src) || bytes % 16 != 0) return VBS_EALIGN;
  int* status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_stateless_status) != cudaSuccess) return VBS_ECUDA;
  return vbs::launch_peak_read(src, bytes, grid, mode, sink, status, reinterpret_cast<cudaStream_t>(stream));
}

// =====================================================================================
// the checked build's bounds-check record
// =====================================================================================

VBS_EXPORT int vbs_checked_record(int* checked, int* site, int64_t* index) {
  if (!checked || !site || !index) return VBS_EINVAL;
#ifdef VBS_CHECKED
  *checked = 1;
#else
  *checked = 0;
#endif
  *site = -1;
  *index = -1;
  if (cudaDeviceSynchronize() != cudaSuccess) return VBS_ECUDA;
  const unsigned long long recs[3] = {vbs::bs_check_record(), vbs::kv_check_record(), vbs::bpd_check_record()};
  for (unsigned long long r : recs) {
    if (r == ~0ull) return VBS_ECUDA;
    if (r && *site < 0) {
      *site = static_cast<int>(r >> 40) - 1;
      *index = static_cast<int64_t>(r & 0xffffffffffull);
    }
  }
  return VBS_OK;
}
