// C-ABI layer of libfa.so: argument checks, rule rewriting, BlockMask buffer layout, tensor-map encoding
// and kernel dispatch. Every check runs on the host before anything is launched.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "fa_launch.h"

namespace fa {

static std::atomic<uint64_t> g_timeout_ns{2000000000ull};

// ------------------------------------------------------------------------------------------------
// Rule rewriting: postfix program -> OR of conjunctions (each conjunction one KV interval, optionally
// intersected with document equality). AND distributes over OR; a conjunction keeps the tightest
// window and prefix bounds.
// ------------------------------------------------------------------------------------------------
struct HTerm {
  bool causal = false, doc = false;
  int64_t win = INT64_MAX, pre = INT64_MAX;
  bool operator==(const HTerm& o) const {
    return causal == o.causal && doc == o.doc && win == o.win && pre == o.pre;
  }
};

static int compile_rule(const fa_mask_rule* r, DevRule* out) {
  if (!r || r->n_ops < 1 || r->n_ops > FA_MAX_RULE_OPS) return FA_ERR_INVALID_ARG;
  std::vector<std::vector<HTerm>> st;
  bool any_doc = false;
  for (int i = 0; i < r->n_ops; ++i) {
    HTerm t;
    switch (r->op[i]) {
      case FA_M_TRUE: st.push_back({t}); break;
      case FA_M_CAUSAL: t.causal = true; st.push_back({t}); break;
      case FA_M_WINDOW: t.win = r->arg[i]; st.push_back({t}); break;
      case FA_M_PREFIX: t.pre = r->arg[i]; st.push_back({t}); break;
      case FA_M_DOC: t.doc = true; any_doc = true; st.push_back({t}); break;
      case FA_M_AND:
      case FA_M_OR: {
        if (st.size() < 2) return FA_ERR_INVALID_ARG;
        std::vector<HTerm> b = st.back();
        st.pop_back();
        std::vector<HTerm> a = st.back();
        st.pop_back();
        std::vector<HTerm> c;
        if (r->op[i] == FA_M_OR) {
          c = a;
          c.insert(c.end(), b.begin(), b.end());
        } else {
          for (const HTerm& x : a)
            for (const HTerm& y : b) {
              HTerm z;
              z.causal = x.causal || y.causal;
              z.doc = x.doc || y.doc;
              z.win = std::min(x.win, y.win);
              z.pre = std::min(x.pre, y.pre);
              c.push_back(z);
            }
        }
        std::vector<HTerm> u;
        for (const HTerm& x : c)
          if (std::find(u.begin(), u.end(), x) == u.end()) u.push_back(x);
        if (u.size() > 64) return FA_ERR_UNSUPPORTED;
        st.push_back(u);
        break;
      }
      default: return FA_ERR_INVALID_ARG;
    }
  }
  if (st.size() != 1) return FA_ERR_INVALID_ARG;
  const std::vector<HTerm>& terms = st.back();
  if (terms.size() > FA_MAX_RULE_TERMS) return FA_ERR_UNSUPPORTED;
  if (any_doc && (!r->doc_ids || r->doc_len < 1 || r->doc_batch < 1)) return FA_ERR_INVALID_ARG;
  if (out) {
    std::memset(out, 0, sizeof(*out));
    out->n_terms = (int32_t)terms.size();
    out->any_doc = 0;
    for (size_t i = 0; i < terms.size(); ++i) {
      out->t[i].causal = terms[i].causal;
      out->t[i].doc = terms[i].doc;
      out->t[i].win = terms[i].win;
      out->t[i].pre = terms[i].pre;
      if (terms[i].doc) out->any_doc = 1;
    }
    out->doc_ids = r->doc_ids;
    out->doc_batch = r->doc_batch;
    out->doc_len = r->doc_len;
    out->q_offset = r->q_offset;
    out->doc_run = nullptr;
    out->doc_sorted = nullptr;
  }
  return FA_OK;
}

static DevScore make_score(const fa_score_rule* s, int kv_len) {
  DevScore d;
  d.alibi = s ? s->alibi_slopes : nullptr;
  d.rel = s ? s->rel_bias : nullptr;
  d.softcap = (s && s->softcap > 0.f) ? s->softcap : 0.f;
  d.inv_softcap = d.softcap > 0.f ? 1.f / d.softcap : 0.f;
  d.kv_len = kv_len;
  return d;
}

static DevMask dev_mask(const fa_block_mask* m) {
  DevMask d;
  d.Bm = m->Bm;
  d.Hm = m->Hm;
  d.q_len = m->q_len;
  d.kv_len = m->kv_len;
  d.bq = m->bq;
  d.bk = m->bk;
  d.nq = m->nq;
  d.nk = m->nk;
  d.kv_num = m->kv_num;
  d.kv_idx = m->kv_idx;
  d.full_kv_num = m->full_kv_num;
  d.full_kv_idx = m->full_kv_idx;
  d.q_num = m->q_num;
  d.q_idx = m->q_idx;
  d.full_q_num = m->full_q_num;
  d.full_q_idx = m->full_q_idx;
  d.row_order = m->row_order;
  return d;
}

// ------------------------------------------------------------------------------------------------
// BlockMask buffer layout
// ------------------------------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct MaskLayout {
  int Bm, Hm, nq, nk;
  size_t off[12];  // the nine tables, document run bounds and sortedness flags (document rules), row order
  size_t total;
};

static bool rule_reads_doc(const fa_mask_rule* r) {
  for (int i = 0; i < r->n_ops && i < FA_MAX_RULE_OPS; ++i)
    if (r->op[i] == FA_M_DOC) return true;
  return false;
}

static int mask_layout(const fa_mask_rule* rule, int B, int H, int Q_LEN, int KV_LEN, int Bq, int Bk,
                       MaskLayout* L) {
  if (!rule) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Q_LEN < 1 || KV_LEN < 1) return FA_ERR_SHAPE;
  if (Bq < 1 || Bq > 128 || Bk < 1 || Bk > 128) return FA_ERR_SHAPE;
  L->Bm = rule->batch_dependent ? B : 1;
  L->Hm = rule->head_dependent ? H : 1;
  L->nq = (Q_LEN + Bq - 1) / Bq;
  L->nk = (KV_LEN + Bk - 1) / Bk;
  const size_t heads = (size_t)L->Bm * L->Hm;
  const size_t rowsz = heads * L->nq * sizeof(int32_t), colsz = heads * L->nk * sizeof(int32_t);
  const size_t grid = heads * (size_t)L->nq * L->nk;
  const bool doc = rule_reads_doc(rule) && rule->doc_len > 0 && rule->doc_batch > 0;
  const size_t nb = doc ? (size_t)rule->doc_batch : 0, dl = doc ? (size_t)rule->doc_len : 0;
  const size_t sizes[12] = {rowsz, rowsz, colsz, colsz, grid * 4, grid * 4, grid * 4, grid * 4, grid,
                            nb * 2 * dl * sizeof(int32_t), nb * sizeof(int32_t), rowsz};
  size_t o = 0;
  for (int i = 0; i < 12; ++i) {
    L->off[i] = o;
    o += align256(sizes[i]);
  }
  L->total = o;
  return FA_OK;
}

// ------------------------------------------------------------------------------------------------
// Tensor maps
// ------------------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

static int encode_tmap(CUtensorMapDataType dt, CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
  if (!enc) return -1;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  CUresult r = enc(m, dt, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

int encode_tmap_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tmap(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, m, base, rank, dims, strides_bytes, box);
}

int encode_tmap_f32(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tmap(CU_TENSOR_MAP_DATA_TYPE_FLOAT32, m, base, rank, dims, strides_bytes, box);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Decode splits of 4096 tokens: long enough that a CTA's start-up (barriers, page-table reads, the first
// copies in flight) is small against its 2 MiB of K/V at d = 128, short enough that the 64-request paged
// decode still runs about 14 waves of CTAs (89.8 % of the measured HBM copy rate against 86.9 % with 2048)
static int decode_pages_per_split(int page, int max_pages) {
  int ps = std::max(1, 4096 / std::max(page, 1));
  return std::min(ps, std::max(max_pages, 1));
}

static int check_forward(const void* q, const void* k, const void* v, const fa_block_mask* bm, void* out,
                         float* lse, int B, int Hq, int Hkv, int Q_LEN, int KV_LEN, int d) {
  if (!q || !k || !v || !bm || !out || !lse) return FA_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Q_LEN < 1 || KV_LEN < 1) return FA_ERR_SHAPE;
  if (Hq % Hkv) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (bm->q_len != Q_LEN || bm->kv_len != KV_LEN) return FA_ERR_SHAPE;  // never trimmed silently
  if (!(bm->Bm == 1 || bm->Bm == B) || !(bm->Hm == 1 || bm->Hm == Hq)) return FA_ERR_SHAPE;
  if (bm->nq != (Q_LEN + bm->bq - 1) / bm->bq || bm->nk != (KV_LEN + bm->bk - 1) / bm->bk) return FA_ERR_SHAPE;
  auto okb = [](int x) { return x == 16 || x == 32 || x == 64 || x == 128; };
  if (!okb(bm->bq) || !okb(bm->bk)) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return FA_ERR_INVALID_ARG;
  if (!bm->kv_num || !bm->kv_idx || !bm->full_kv_num || !bm->full_kv_idx) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

struct PagedKV {  // all zero: contiguous K / V
  const int32_t* page_table;
  int32_t n_pages_total, page, max_pages;
};

// Split rows: the derived tables (entries e = r * ncm + c) and the per-entry outputs the forward writes
// instead of O and LSE.
struct SplitPlan {
  DevMask mask;
  int32_t ncm;
  float* o_part;    // fp32 [B, Hq, nq * ncm * 128, d]
  float* lse_part;  // fp32 [B, Hq, nq * ncm * 128]
};

static int forward_impl(bool force_mma, const void* q, const void* k, const void* v, const fa_block_mask* bm,
                        const fa_score_rule* score, float scale, void* out, int32_t out_dtype, float* lse,
                        int32_t B, int32_t Hq,
                        int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN, int32_t d, int32_t* dev_status,
                        int64_t* dev_counters, fa_stream_t stream, const PagedKV& pg = PagedKV{},
                        const SplitPlan* split = nullptr) {
  int s = check_forward(q, k, v, bm, out, lse, B, Hq, Hkv, Q_LEN, KV_LEN, d);
  if (s != FA_OK) return s;
  if (out_dtype != FA_OUT_BF16 && out_dtype != FA_OUT_F32) return FA_ERR_INVALID_ARG;
  if (pg.page_table) {  // one page per key block; the table covers every key block
    if (pg.page != bm->bk || pg.n_pages_total < 1 || pg.max_pages < bm->nk) return FA_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(pg.page_table) & 3u) return FA_ERR_INVALID_ARG;
  }
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  s = compile_rule(&bm->rule, &a.rule);
  a.rule.doc_run = bm->doc_run;
  a.rule.doc_sorted = bm->doc_sorted;
  if (s != FA_OK) return s;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.out_f32 = out_dtype == FA_OUT_F32;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.q_len = Q_LEN;
  a.kv_len = KV_LEN;
  a.d = d;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt((float)d);
  a.score = make_score(score, KV_LEN);
  a.mask = dev_mask(bm);
  a.status = dev_status;
  a.counters = dev_counters;
  a.timeout_ns = g_timeout_ns.load();
  a.page_table = pg.page_table;
  a.max_pages = pg.max_pages;
  a.n_pages_total = pg.n_pages_total;
  a.split_ncm = 1;
  a.out_q_len = Q_LEN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (split) {  // the tcgen05 kernel over the derived tables, writing each entry's O and LSE
    a.mask = split->mask;
    a.split_ncm = split->ncm;
    a.out_q_len = split->mask.nq * 128;
    a.out = split->o_part;
    a.out_f32 = 1;
    a.lse = split->lse_part;
    return launch_fwd_tc5(a, st);
  }
  if (!force_mma && bm->bq == 128 && bm->bk == 128) {
    int r = launch_fwd_tc5(a, st);
    if (r != FA_ERR_UNSUPPORTED) return r;
  }
  return launch_fwd_mma(a, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

static int backward_impl(const void* q, const void* k, const void* v, const void* out, int32_t out_dtype,
                         const void* dout, const float* lse, const fa_block_mask* bm, const fa_score_rule* score,
                         float scale, float* dq, float* dk, float* dv, float* delta, int32_t B, int32_t Hq,
                         int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN, int32_t d, int32_t* dev_status,
                         fa_stream_t stream) {
  if (!dout || !dq || !dk || !dv || !delta) return FA_ERR_INVALID_ARG;
  int s = check_forward(q, k, v, bm, const_cast<void*>(out), const_cast<float*>(lse), B, Hq, Hkv, Q_LEN, KV_LEN, d);
  if (s != FA_OK) return s;
  if (out_dtype != FA_OUT_BF16 && out_dtype != FA_OUT_F32) return FA_ERR_INVALID_ARG;
  if ((bm->bq != 64 && bm->bq != 128) || (bm->bk != 64 && bm->bk != 128)) return FA_ERR_UNSUPPORTED;
  if (!bm->q_num || !bm->q_idx || !bm->full_q_num || !bm->full_q_idx) return FA_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv)) return FA_ERR_INVALID_ARG;
  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  s = compile_rule(&bm->rule, &a.rule);
  if (s != FA_OK) return s;
  a.rule.doc_run = bm->doc_run;
  a.rule.doc_sorted = bm->doc_sorted;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.out_f32 = out_dtype == FA_OUT_F32;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.delta = delta;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.q_len = Q_LEN;
  a.kv_len = KV_LEN;
  a.d = d;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt((float)d);
  a.score = make_score(score, KV_LEN);
  a.mask = dev_mask(bm);
  a.status = dev_status;
  a.timeout_ns = g_timeout_ns.load();
  if ((long long)B * Hq > 65535LL * 65535LL || Hq > 65535 || B > 65535) return FA_ERR_UNSUPPORTED;
  return launch_backward(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_SHAPE: return "inconsistent shapes";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device wait timed out";
    case FA_ERR_DEVICE_CHECK: return "device-side index check failed";
    case FA_ERR_BUFFER_TOO_SMALL: return "buffer too small";
  }
  return "unknown status";
}

const char* fa_version(void) { return "libfa 0.1 sm_103a"; }

void fa_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }
uint64_t fa_get_wait_timeout_ns(void) { return g_timeout_ns.load(); }

size_t fa_block_mask_bytes(const fa_mask_rule* rule, int32_t B, int32_t H, int32_t Q_LEN, int32_t KV_LEN,
                           int32_t Bq, int32_t Bk) {
  MaskLayout L;
  if (mask_layout(rule, B, H, Q_LEN, KV_LEN, Bq, Bk, &L) != FA_OK) return 0;
  return L.total;
}

fa_status fa_create_block_mask(const fa_mask_rule* rule, int32_t B, int32_t H, int32_t Q_LEN, int32_t KV_LEN,
                               int32_t Bq, int32_t Bk, void* dev_buf, size_t buf_bytes, fa_block_mask* out,
                               fa_stream_t stream) {
  if (!rule || !out || !dev_buf) return FA_ERR_INVALID_ARG;
  MaskLayout L;
  int s = mask_layout(rule, B, H, Q_LEN, KV_LEN, Bq, Bk, &L);
  if (s != FA_OK) return (fa_status)s;
  if (buf_bytes < L.total) return FA_ERR_BUFFER_TOO_SMALL;
  if (reinterpret_cast<uintptr_t>(dev_buf) & 255u) return FA_ERR_INVALID_ARG;
  DevRule R;
  s = compile_rule(rule, &R);
  if (s != FA_OK) return (fa_status)s;
  // per-batch state (document layouts per b, per-request query offsets) needs a per-batch table
  const bool per_b_state = (R.any_doc && rule->doc_batch > 1) || rule->q_offset != nullptr;
  if (per_b_state && !rule->batch_dependent && B > 1) return FA_ERR_INVALID_ARG;
  if (R.any_doc && (rule->doc_batch != 1 && rule->doc_batch != B)) return FA_ERR_SHAPE;
  if (R.any_doc && rule->doc_len < KV_LEN) return FA_ERR_SHAPE;
  uint8_t* base = static_cast<uint8_t*>(dev_buf);
  MaskOut T;
  T.Bm = L.Bm;
  T.Hm = L.Hm;
  T.q_len = Q_LEN;
  T.kv_len = KV_LEN;
  T.bq = Bq;
  T.bk = Bk;
  T.nq = L.nq;
  T.nk = L.nk;
  T.kv_num = reinterpret_cast<int32_t*>(base + L.off[0]);
  T.full_kv_num = reinterpret_cast<int32_t*>(base + L.off[1]);
  T.q_num = reinterpret_cast<int32_t*>(base + L.off[2]);
  T.full_q_num = reinterpret_cast<int32_t*>(base + L.off[3]);
  T.kv_idx = reinterpret_cast<int32_t*>(base + L.off[4]);
  T.full_kv_idx = reinterpret_cast<int32_t*>(base + L.off[5]);
  T.q_idx = reinterpret_cast<int32_t*>(base + L.off[6]);
  T.full_q_idx = reinterpret_cast<int32_t*>(base + L.off[7]);
  T.block_class = base + L.off[8];
  T.doc_run = R.any_doc ? reinterpret_cast<int32_t*>(base + L.off[9]) : nullptr;
  T.doc_sorted = R.any_doc ? reinterpret_cast<int32_t*>(base + L.off[10]) : nullptr;
  T.row_order = L.nq > 1 ? reinterpret_cast<int32_t*>(base + L.off[11]) : nullptr;  // one row: nothing to order
  if (L.Hm > 65535 || L.Bm > 65535 || L.nq > INT_MAX / 2 || L.nk > 65535 * 1024) return FA_ERR_UNSUPPORTED;
  if (launch_mask_build(R, T, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  out->Bm = T.Bm;
  out->Hm = T.Hm;
  out->q_len = Q_LEN;
  out->kv_len = KV_LEN;
  out->bq = Bq;
  out->bk = Bk;
  out->nq = T.nq;
  out->nk = T.nk;
  out->kv_num = T.kv_num;
  out->kv_idx = T.kv_idx;
  out->full_kv_num = T.full_kv_num;
  out->full_kv_idx = T.full_kv_idx;
  out->q_num = T.q_num;
  out->q_idx = T.q_idx;
  out->full_q_num = T.full_q_num;
  out->full_q_idx = T.full_q_idx;
  out->block_class = T.block_class;
  out->doc_run = T.doc_run;
  out->doc_sorted = T.doc_sorted;
  out->row_order = T.row_order;
  out->rule = *rule;
  return FA_OK;
}

// Layout of the one-row-per-request mask fa_block_mask_select_rows writes: Bm = Bz, Hm = src->Hm, nq = 1.
static int select_layout(const fa_block_mask* src, int32_t Bz, MaskLayout* L) {
  if (!src || Bz < 1) return FA_ERR_INVALID_ARG;
  if (src->nq < 1 || src->nk < 1 || src->Hm < 1 || src->bk < 1) return FA_ERR_SHAPE;
  if (src->Bm != 1 && src->Bm != Bz) return FA_ERR_SHAPE;
  fa_mask_rule r;
  std::memset(&r, 0, sizeof(r));
  r.n_ops = 1;
  r.op[0] = FA_M_TRUE;
  r.batch_dependent = 1;
  r.head_dependent = src->Hm > 1;
  return mask_layout(&r, Bz, src->Hm, 1, src->kv_len, 1, src->bk, L);
}

size_t fa_block_mask_select_bytes(const fa_block_mask* src, int32_t Bz) {
  MaskLayout L;
  return select_layout(src, Bz, &L) == FA_OK ? L.total : 0;
}

fa_status fa_block_mask_select_rows(const fa_block_mask* src, const int32_t* dev_q_pos, int32_t Bz, void* dev_buf,
                                    size_t buf_bytes, fa_block_mask* out, int32_t* dev_status, fa_stream_t stream) {
  if (!src || !dev_q_pos || !dev_buf || !out) return FA_ERR_INVALID_ARG;
  if (src->rule.q_offset) return FA_ERR_INVALID_ARG;  // the prebuilt table must be in global positions
  if (!src->kv_num || !src->kv_idx || !src->full_kv_num || !src->full_kv_idx || !src->block_class)
    return FA_ERR_INVALID_ARG;
  MaskLayout L;
  int s = select_layout(src, Bz, &L);
  if (s != FA_OK) return (fa_status)s;
  if (buf_bytes < L.total) return FA_ERR_BUFFER_TOO_SMALL;
  if (reinterpret_cast<uintptr_t>(dev_buf) & 255u) return FA_ERR_INVALID_ARG;
  if (Bz > 65535 || src->Hm > 65535) return FA_ERR_UNSUPPORTED;
  MaskOut S;
  std::memset(&S, 0, sizeof(S));
  S.Bm = src->Bm;
  S.Hm = src->Hm;
  S.q_len = src->q_len;
  S.kv_len = src->kv_len;
  S.bq = src->bq;
  S.bk = src->bk;
  S.nq = src->nq;
  S.nk = src->nk;
  S.kv_num = src->kv_num;
  S.kv_idx = src->kv_idx;
  S.full_kv_num = src->full_kv_num;
  S.full_kv_idx = src->full_kv_idx;
  S.block_class = src->block_class;
  uint8_t* base = static_cast<uint8_t*>(dev_buf);
  MaskOut D;
  std::memset(&D, 0, sizeof(D));
  D.Bm = Bz;
  D.Hm = src->Hm;
  D.q_len = 1;
  D.kv_len = src->kv_len;
  D.bq = 1;
  D.bk = src->bk;
  D.nq = 1;
  D.nk = src->nk;
  D.kv_num = reinterpret_cast<int32_t*>(base + L.off[0]);
  D.full_kv_num = reinterpret_cast<int32_t*>(base + L.off[1]);
  D.q_num = reinterpret_cast<int32_t*>(base + L.off[2]);
  D.full_q_num = reinterpret_cast<int32_t*>(base + L.off[3]);
  D.kv_idx = reinterpret_cast<int32_t*>(base + L.off[4]);
  D.full_kv_idx = reinterpret_cast<int32_t*>(base + L.off[5]);
  D.q_idx = reinterpret_cast<int32_t*>(base + L.off[6]);
  D.full_q_idx = reinterpret_cast<int32_t*>(base + L.off[7]);
  D.block_class = base + L.off[8];
  DevRule R;
  s = compile_rule(&src->rule, &R);
  if (s != FA_OK) return (fa_status)s;
  R.q_offset = dev_q_pos;
  R.doc_run = src->doc_run;
  R.doc_sorted = src->doc_sorted;
  if (R.any_doc && src->rule.doc_batch != 1 && src->rule.doc_batch != Bz) return FA_ERR_SHAPE;
  if (launch_mask_select(R, S, Bz, D, dev_status, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  out->Bm = D.Bm;
  out->Hm = D.Hm;
  out->q_len = 1;
  out->kv_len = D.kv_len;
  out->bq = 1;
  out->bk = D.bk;
  out->nq = 1;
  out->nk = D.nk;
  out->kv_num = D.kv_num;
  out->kv_idx = D.kv_idx;
  out->full_kv_num = D.full_kv_num;
  out->full_kv_idx = D.full_kv_idx;
  out->q_num = D.q_num;
  out->q_idx = D.q_idx;
  out->full_q_num = D.full_q_num;
  out->full_q_idx = D.full_q_idx;
  out->block_class = D.block_class;
  out->doc_run = src->doc_run;  // same document ids, same runs
  out->doc_sorted = src->doc_sorted;
  out->row_order = nullptr;  // one row per request
  out->rule = src->rule;
  out->rule.q_offset = dev_q_pos;  // the one query row of request b sits at global position q_pos[b]
  out->rule.batch_dependent = 1;
  return FA_OK;
}

fa_status fa_flex_forward(const void* q, const void* k, const void* v, const fa_block_mask* block_mask,
                          const fa_score_rule* score_rule, float scale, void* out, int32_t out_dtype, float* lse,
                          int32_t B, int32_t Hq, int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN, int32_t d,
                          int32_t* dev_status, int64_t* dev_counters, fa_stream_t stream) {
  return (fa_status)forward_impl(false, q, k, v, block_mask, score_rule, scale, out, out_dtype, lse, B, Hq, Hkv, Q_LEN,
                                 KV_LEN, d, dev_status, dev_counters, stream);
}

fa_status fa_flex_forward_paged(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                                int32_t n_pages_total, int32_t page, int32_t max_pages,
                                const fa_block_mask* block_mask, const fa_score_rule* score_rule, float scale,
                                void* out, int32_t out_dtype, float* lse, int32_t B, int32_t Hq, int32_t Hkv,
                                int32_t Q_LEN, int32_t KV_LEN, int32_t d, int32_t* dev_status, fa_stream_t stream) {
  if (!page_table) return FA_ERR_INVALID_ARG;
  return (fa_status)forward_impl(false, q, k_pages, v_pages, block_mask, score_rule, scale, out, out_dtype, lse, B,
                                 Hq, Hkv, Q_LEN, KV_LEN, d, dev_status, nullptr, stream,
                                 PagedKV{page_table, n_pages_total, page, max_pages});
}

// ------------------------------------------------------------------------------------------------
// Forward from host buffers: chunks of KV heads of one batch row stream through two device slots; the
// copies in, the kernels (two streams, so a chunk's CTAs can fill the SMs the previous chunk's short CTAs
// free) and the copies out run on separate streams, so each chunk's copies overlap its neighbours' work.
// ------------------------------------------------------------------------------------------------
// The host path streams about kHostChunks chunks (whole KV heads of one batch row each) through
// kHostSlots device buffers: a chunk's copies in wait only for the copies out of the chunk kHostSlots
// earlier. Measured on cfg2 (201 MB in, 135 MB out, 1.14 ms for the copies alone in both directions): 3
// slots x 8 chunks 1.40 ms, 2 x 8 1.47 ms, 4 x 8 and 3 x 4 1.40 ms, 3 x 16 1.46 ms, 3 x 32 1.77 ms (smaller
// copies run below the link's rate).
constexpr int kHostSlots = 3;
constexpr int kHostChunks = 8;
struct HostPlan {
  int ck, g, n_chunks, chunks_per_b, n_slots;
  size_t q_bytes, kv_bytes, o_bytes, l_bytes, slot_bytes;
};

static int host_plan(int B, int Hq, int Hkv, int Q_LEN, int KV_LEN, int d, int out_dtype, HostPlan* P) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Q_LEN < 1 || KV_LEN < 1 || Hq % Hkv) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (out_dtype != FA_OUT_BF16 && out_dtype != FA_OUT_F32) return FA_ERR_INVALID_ARG;
  P->g = Hq / Hkv;
  const int units = B * Hkv;
  P->ck = std::max(1, std::min(Hkv, units / kHostChunks));
  P->chunks_per_b = (Hkv + P->ck - 1) / P->ck;
  P->n_chunks = B * P->chunks_per_b;
  P->n_slots = std::min(kHostSlots, P->n_chunks);
  const size_t qh = (size_t)Q_LEN * d, kh = (size_t)KV_LEN * d;
  P->q_bytes = align256((size_t)P->ck * P->g * qh * 2);
  P->kv_bytes = align256((size_t)P->ck * kh * 2);
  P->o_bytes = align256((size_t)P->ck * P->g * qh * (out_dtype == FA_OUT_F32 ? 4 : 2));
  P->l_bytes = align256((size_t)P->ck * P->g * Q_LEN * 4);
  P->slot_bytes = P->q_bytes + 2 * P->kv_bytes + P->o_bytes + P->l_bytes;
  return FA_OK;
}

size_t fa_forward_host_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN, int32_t d,
                                       int32_t out_dtype) {
  HostPlan P;
  return host_plan(B, Hq, Hkv, Q_LEN, KV_LEN, d, out_dtype, &P) == FA_OK ? P.n_slots * P.slot_bytes : 0;
}

fa_status fa_flex_forward_host(const void* host_q, const void* host_k, const void* host_v,
                               const fa_block_mask* block_mask, const fa_score_rule* score_rule, float scale,
                               void* host_out, int32_t out_dtype, float* host_lse, int32_t B, int32_t Hq, int32_t Hkv,
                               int32_t Q_LEN, int32_t KV_LEN, int32_t d, void* dev_workspace, size_t workspace_bytes,
                               int32_t* dev_status, fa_stream_t stream) {
  if (!host_q || !host_k || !host_v || !block_mask || !host_out || !host_lse || !dev_workspace)
    return FA_ERR_INVALID_ARG;
  HostPlan P;
  int s = host_plan(B, Hq, Hkv, Q_LEN, KV_LEN, d, out_dtype, &P);
  if (s != FA_OK) return (fa_status)s;
  if (workspace_bytes < P.n_slots * P.slot_bytes) return FA_ERR_BUFFER_TOO_SMALL;
  if (reinterpret_cast<uintptr_t>(dev_workspace) & 255u) return FA_ERR_INVALID_ARG;
  const fa_block_mask& M = *block_mask;
  if (M.q_len != Q_LEN || M.kv_len != KV_LEN || !(M.Bm == 1 || M.Bm == B) || !(M.Hm == 1 || M.Hm == Hq))
    return FA_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t s_in = nullptr, s_out = nullptr, s_c1 = nullptr;
  cudaEvent_t ev_start = nullptr, ev_in[kHostSlots] = {}, ev_done[kHostSlots] = {}, ev_free[kHostSlots] = {};
  bool cuda_ok = cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaStreamCreateWithFlags(&s_c1, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; i < P.n_slots && cuda_ok; ++i)
    cuda_ok = cudaEventCreateWithFlags(&ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&ev_done[i], cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&ev_free[i], cudaEventDisableTiming) == cudaSuccess;
  // the side streams start after everything already queued on `stream` (e.g. the mask build)
  if (cuda_ok) cuda_ok = cudaEventRecord(ev_start, st) == cudaSuccess && cudaStreamWaitEvent(s_in, ev_start, 0) ==
                         cudaSuccess && cudaStreamWaitEvent(s_out, ev_start, 0) == cudaSuccess &&
                         cudaStreamWaitEvent(s_c1, ev_start, 0) == cudaSuccess;
  const size_t qh = (size_t)Q_LEN * d, kh = (size_t)KV_LEN * d;
  const size_t oel = out_dtype == FA_OUT_F32 ? 4 : 2;
  int status = cuda_ok ? FA_OK : FA_ERR_CUDA;
  for (int c = 0; c < P.n_chunks && status == FA_OK; ++c) {
    const int slot = c % P.n_slots;
    cudaStream_t sc = (c & 1) ? s_c1 : st;  // the chunk's kernels (two streams, so that they may overlap)
    const int b = c / P.chunks_per_b, hk0 = (c % P.chunks_per_b) * P.ck;
    const int nk = std::min(P.ck, Hkv - hk0), h0 = hk0 * P.g, nq = nk * P.g;
    uint8_t* base = static_cast<uint8_t*>(dev_workspace) + slot * P.slot_bytes;
    void* dq = base;
    void* dk = base + P.q_bytes;
    void* dv = base + P.q_bytes + P.kv_bytes;
    void* dout = base + P.q_bytes + 2 * P.kv_bytes;
    float* dlse = reinterpret_cast<float*>(base + P.q_bytes + 2 * P.kv_bytes + P.o_bytes);
    // copies in, once the copies out of the chunk that used this slot before have finished
    if (c >= P.n_slots && cudaStreamWaitEvent(s_in, ev_free[slot], 0) != cudaSuccess) { status = FA_ERR_CUDA; break; }
    const size_t qoff = ((size_t)b * Hq + h0) * qh, koff = ((size_t)b * Hkv + hk0) * kh;
    if (cudaMemcpyAsync(dq, static_cast<const uint8_t*>(host_q) + qoff * 2, (size_t)nq * qh * 2,
                        cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
        cudaMemcpyAsync(dk, static_cast<const uint8_t*>(host_k) + koff * 2, (size_t)nk * kh * 2,
                        cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
        cudaMemcpyAsync(dv, static_cast<const uint8_t*>(host_v) + koff * 2, (size_t)nk * kh * 2,
                        cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
        cudaEventRecord(ev_in[slot], s_in) != cudaSuccess || cudaStreamWaitEvent(sc, ev_in[slot], 0) != cudaSuccess) {
      status = FA_ERR_CUDA;
      break;
    }
    // the chunk's view of the mask, the rules and the score: batch row b, heads h0 .. h0 + nq - 1
    fa_block_mask V = M;
    size_t row0 = 0;
    if (M.Bm > 1) row0 += (size_t)b * M.Hm * M.nq;
    if (M.Hm > 1) row0 += (size_t)h0 * M.nq;
    V.Bm = 1;
    V.Hm = M.Hm > 1 ? nq : 1;
    V.kv_num = M.kv_num + row0;
    V.full_kv_num = M.full_kv_num + row0;
    V.kv_idx = M.kv_idx + row0 * M.nk;
    V.full_kv_idx = M.full_kv_idx + row0 * M.nk;
    V.q_num = V.q_idx = V.full_q_num = V.full_q_idx = nullptr;  // the forward reads the row tables only
    V.block_class = M.block_class ? M.block_class + row0 * M.nk : nullptr;
    V.row_order = M.row_order ? M.row_order + row0 : nullptr;
    if (M.rule.q_offset) V.rule.q_offset = M.rule.q_offset + (M.Bm > 1 ? b : 0);
    if (M.rule.doc_ids && M.rule.doc_batch > 1) {
      V.rule.doc_ids = M.rule.doc_ids + (size_t)b * M.rule.doc_len;
      V.rule.doc_batch = 1;
      if (M.doc_run) V.doc_run = M.doc_run + (size_t)b * 2 * M.rule.doc_len;
      if (M.doc_sorted) V.doc_sorted = M.doc_sorted + b;
    }
    fa_score_rule S;
    const fa_score_rule* Sp = nullptr;
    if (score_rule) {
      S = *score_rule;
      if (S.alibi_slopes) S.alibi_slopes += h0;
      if (S.rel_bias) S.rel_bias += (size_t)h0 * (2 * (size_t)KV_LEN - 1);
      Sp = &S;
    }
    s = forward_impl(false, dq, dk, dv, &V, Sp, scale, dout, out_dtype, dlse, 1, nq, nk, Q_LEN, KV_LEN, d, dev_status,
                     nullptr, reinterpret_cast<fa_stream_t>(sc));
    if (s != FA_OK) { status = s; break; }
    // copies out
    if (cudaEventRecord(ev_done[slot], sc) != cudaSuccess || cudaStreamWaitEvent(s_out, ev_done[slot], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint8_t*>(host_out) + qoff * oel, dout, (size_t)nq * qh * oel,
                        cudaMemcpyDeviceToHost, s_out) != cudaSuccess ||
        cudaMemcpyAsync(host_lse + ((size_t)b * Hq + h0) * Q_LEN, dlse, (size_t)nq * Q_LEN * 4, cudaMemcpyDeviceToHost,
                        s_out) != cudaSuccess ||
        cudaEventRecord(ev_free[slot], s_out) != cudaSuccess) {
      status = FA_ERR_CUDA;
      break;
    }
  }
  // `stream` completes after the last copy out; the side streams and events are released when idle
  if (s_out && cudaEventRecord(ev_start, s_out) == cudaSuccess) cudaStreamWaitEvent(st, ev_start, 0);
  if (s_c1 && ev_in[0] && cudaEventRecord(ev_in[0], s_c1) == cudaSuccess) cudaStreamWaitEvent(st, ev_in[0], 0);
  for (int i = 0; i < kHostSlots; ++i) {
    if (ev_in[i]) cudaEventDestroy(ev_in[i]);
    if (ev_done[i]) cudaEventDestroy(ev_done[i]);
    if (ev_free[i]) cudaEventDestroy(ev_free[i]);
  }
  if (ev_start) cudaEventDestroy(ev_start);
  if (s_in) cudaStreamDestroy(s_in);
  if (s_out) cudaStreamDestroy(s_out);
  if (s_c1) cudaStreamDestroy(s_c1);
  return (fa_status)status;
}

fa_status fa_flex_forward_mma(const void* q, const void* k, const void* v, const fa_block_mask* block_mask,
                              const fa_score_rule* score_rule, float scale, void* out, int32_t out_dtype,
                              float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN,
                              int32_t d, int32_t* dev_status, int64_t* dev_counters, fa_stream_t stream) {
  return (fa_status)forward_impl(true, q, k, v, block_mask, score_rule, scale, out, out_dtype, lse, B, Hq, Hkv, Q_LEN,
                                 KV_LEN, d, dev_status, dev_counters, stream);
}

fa_status fa_flex_backward(const void* q, const void* k, const void* v, const void* out, int32_t out_dtype,
                           const void* dout, const float* lse, const fa_block_mask* block_mask,
                           const fa_score_rule* score_rule, float scale, float* dq, float* dk, float* dv,
                           float* delta, int32_t B, int32_t Hq, int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN, int32_t d,
                           int32_t* dev_status, fa_stream_t stream) {
  return (fa_status)backward_impl(q, k, v, out, out_dtype, dout, lse, block_mask, score_rule, scale, dq, dk, dv, delta,
                                  B, Hq, Hkv, Q_LEN, KV_LEN, d, dev_status, stream);
}

size_t fa_decode_workspace_bytes(int32_t Bz, int32_t Hq, int32_t d, int32_t max_pages, int32_t page) {
  if (Bz < 1 || Hq < 1 || d < 1 || max_pages < 1 || page < 1) return 0;
  const int ps = decode_pages_per_split(page, max_pages);
  const size_t ns = (size_t)((max_pages + ps - 1) / ps);
  const size_t slots = (size_t)Bz * Hq * ns;
  return align256(slots * 4) * 3 + align256(slots * (size_t)d * 4);
}

fa_status fa_flex_decode(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                         int32_t n_pages_total, const fa_block_mask* bm, const fa_score_rule* score_rule,
                         float scale, void* out, int32_t out_dtype, float* lse, int32_t Bz, int32_t Hq, int32_t Hkv,
                         int32_t d,
                         int32_t page, int32_t max_pages, void* workspace, size_t workspace_bytes,
                         int32_t* dev_status, int64_t* dev_counters, fa_stream_t stream) {
  if (!q || !k_pages || !v_pages || !page_table || !bm || !out || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (Bz < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || n_pages_total < 1 || max_pages < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (page != 32 && page != 64 && page != 128) return FA_ERR_UNSUPPORTED;
  if (out_dtype != FA_OUT_BF16 && out_dtype != FA_OUT_F32) return FA_ERR_INVALID_ARG;
  if (Hq / Hkv > 16) return FA_ERR_UNSUPPORTED;
  if (bm->bq != 1 || bm->bk != page || bm->q_len != 1 || (int64_t)bm->kv_len != (int64_t)max_pages * page ||
      bm->Hm != 1 || !(bm->Bm == 1 || bm->Bm == Bz) || bm->nk != max_pages || bm->nq != 1)
    return FA_ERR_SHAPE;
  if ((int64_t)n_pages_total * Hkv * page > INT_MAX) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(workspace))
    return FA_ERR_INVALID_ARG;
  const size_t need = fa_decode_workspace_bytes(Bz, Hq, d, max_pages, page);
  if (workspace_bytes < need) return FA_ERR_BUFFER_TOO_SMALL;
  DecArgs a;
  std::memset(&a, 0, sizeof(a));
  int s = compile_rule(&bm->rule, &a.rule);
  a.rule.doc_run = bm->doc_run;
  a.rule.doc_sorted = bm->doc_sorted;
  if (s != FA_OK) return (fa_status)s;
  a.q = q;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.page_table = page_table;
  a.n_pages_total = n_pages_total;
  a.out = out;
  a.out_f32 = out_dtype == FA_OUT_F32;
  a.lse = lse;
  a.Bz = Bz;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.page = page;
  a.max_pages = max_pages;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt((float)d);
  a.score = make_score(score_rule, bm->kv_len);
  a.mask = dev_mask(bm);
  a.pages_per_split = decode_pages_per_split(page, max_pages);
  a.n_splits = (max_pages + a.pages_per_split - 1) / a.pages_per_split;
  const size_t slots = (size_t)Bz * Hq * a.n_splits;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  a.ws_m = reinterpret_cast<float*>(w);
  a.ws_l = reinterpret_cast<float*>(w + align256(slots * 4));
  a.ws_le = reinterpret_cast<float*>(w + 2 * align256(slots * 4));
  a.ws_u = reinterpret_cast<float*>(w + 3 * align256(slots * 4));
  a.status = dev_status;
  a.counters = dev_counters;
  a.timeout_ns = g_timeout_ns.load();
  return (fa_status)launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------------------------------------
// Split rows ("5 Kernels ...", section 5)
// ------------------------------------------------------------------------------------------------
struct SplitLayout {
  int ncm;
  size_t nqd, off_num, off_fnum, off_order, off_idx, off_fidx, off_o, off_lse, total;
};

static bool split_layout(const fa_block_mask* bm, int32_t B, int32_t Hq, int32_t d, int32_t C, SplitLayout* L) {
  if (!bm || B < 1 || Hq < 1 || d < 1 || C < 1 || bm->nq < 1 || bm->nk < 1) return false;
  L->ncm = (bm->nk + C - 1) / C;
  L->nqd = (size_t)bm->nq * L->ncm;
  if (L->nqd * 128 > (size_t)INT_MAX) return false;
  const size_t bh = (size_t)bm->Bm * bm->Hm, rows = (size_t)B * Hq * L->nqd * 128;
  size_t o = 0;
  L->off_num = o;   o += align256(bh * L->nqd * 4);
  L->off_fnum = o;  o += align256(bh * L->nqd * 4);
  L->off_order = o; o += align256(bh * L->nqd * 4);
  L->off_idx = o;   o += align256(bh * L->nqd * C * 4);
  L->off_fidx = o;  o += align256(bh * L->nqd * C * 4);
  L->off_o = o;     o += align256(rows * d * 4);
  L->off_lse = o;   o += align256(rows * 4);
  L->total = o;
  return true;
}

size_t fa_forward_split_workspace_bytes(const fa_block_mask* bm, int32_t B, int32_t Hq, int32_t d,
                                        int32_t chunk_blocks) {
  SplitLayout L;
  return split_layout(bm, B, Hq, d, chunk_blocks, &L) ? L.total : 0;
}

fa_status fa_flex_forward_split(const void* q, const void* k, const void* v, const fa_block_mask* bm,
                                const fa_score_rule* score_rule, float scale, void* out, int32_t out_dtype,
                                float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN,
                                int32_t d, int32_t chunk_blocks, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, fa_stream_t stream) {
  int s = check_forward(q, k, v, bm, out, lse, B, Hq, Hkv, Q_LEN, KV_LEN, d);
  if (s != FA_OK) return (fa_status)s;
  if (out_dtype != FA_OUT_BF16 && out_dtype != FA_OUT_F32) return FA_ERR_INVALID_ARG;
  if (bm->bq != 128 || bm->bk != 128) return FA_ERR_UNSUPPORTED;
  if (chunk_blocks < 1 || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FA_ERR_INVALID_ARG;
  SplitLayout L;
  if (!split_layout(bm, B, Hq, d, chunk_blocks, &L)) return FA_ERR_SHAPE;
  if (workspace_bytes < L.total) return FA_ERR_BUFFER_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  MaskOut S;
  std::memset(&S, 0, sizeof(S));
  S.Bm = bm->Bm;
  S.Hm = bm->Hm;
  S.nq = bm->nq;
  S.nk = bm->nk;
  S.kv_num = bm->kv_num;
  S.kv_idx = bm->kv_idx;
  S.full_kv_num = bm->full_kv_num;
  S.full_kv_idx = bm->full_kv_idx;
  MaskOut D;
  std::memset(&D, 0, sizeof(D));
  D.Bm = bm->Bm;
  D.Hm = bm->Hm;
  D.q_len = Q_LEN;
  D.kv_len = KV_LEN;
  D.bq = D.bk = 128;
  D.nq = (int32_t)L.nqd;
  D.nk = chunk_blocks;  // row stride of the derived lists
  D.kv_num = reinterpret_cast<int32_t*>(w + L.off_num);
  D.full_kv_num = reinterpret_cast<int32_t*>(w + L.off_fnum);
  D.row_order = reinterpret_cast<int32_t*>(w + L.off_order);
  D.kv_idx = reinterpret_cast<int32_t*>(w + L.off_idx);
  D.full_kv_idx = reinterpret_cast<int32_t*>(w + L.off_fidx);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (launch_mask_split(S, chunk_blocks, L.ncm, D, st) != cudaSuccess) return FA_ERR_CUDA;
  SplitPlan P;
  std::memset(&P, 0, sizeof(P));
  P.mask.Bm = D.Bm;
  P.mask.Hm = D.Hm;
  P.mask.q_len = Q_LEN;
  P.mask.kv_len = KV_LEN;
  P.mask.bq = P.mask.bk = 128;
  P.mask.nq = D.nq;
  P.mask.nk = D.nk;
  P.mask.kv_num = D.kv_num;
  P.mask.kv_idx = D.kv_idx;
  P.mask.full_kv_num = D.full_kv_num;
  P.mask.full_kv_idx = D.full_kv_idx;
  P.mask.row_order = D.row_order;
  P.ncm = L.ncm;
  P.o_part = reinterpret_cast<float*>(w + L.off_o);
  P.lse_part = reinterpret_cast<float*>(w + L.off_lse);
  s = forward_impl(false, q, k, v, bm, score_rule, scale, out, out_dtype, lse, B, Hq, Hkv, Q_LEN, KV_LEN, d,
                   dev_status, nullptr, stream, PagedKV{}, &P);
  if (s != FA_OK) return (fa_status)s;
  return launch_split_combine(P.o_part, P.lse_part, B, Hq, Q_LEN, bm->nq, L.ncm, d, out, out_dtype == FA_OUT_F32,
                              lse, st) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status fa_block_mask_stats(const fa_block_mask* bm, int64_t* dev_out, fa_stream_t stream) {
  if (!bm || !dev_out || !bm->kv_num || !bm->full_kv_num) return FA_ERR_INVALID_ARG;
  MaskOut T;
  std::memset(&T, 0, sizeof(T));
  T.Bm = bm->Bm;
  T.Hm = bm->Hm;
  T.nq = bm->nq;
  T.nk = bm->nk;
  T.kv_num = bm->kv_num;
  T.full_kv_num = bm->full_kv_num;
  return launch_mask_stats(T, dev_out, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                                : FA_ERR_CUDA;
}

fa_status fa_check_status(const int32_t* dev_status, fa_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  if (!dev_status) return FA_OK;
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, dev_status, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  return (fa_status)h;
}

fa_status fa_debug_wait_timeout(int32_t* dev_status, uint64_t timeout_ns, fa_stream_t stream) {
  if (!dev_status) return FA_ERR_INVALID_ARG;
  return launch_debug_wait(dev_status, timeout_ns ? timeout_ns : 1, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

}  // extern "C"
