// C-ABI runtime of the DFlash draft-pass library: handle, validation,
// workspace plan and the launch sequence of each entry point.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/dflash.h"
#include "../../include/dflash_testing.h"
#include "kernels.h"

using namespace dflash;

namespace {

thread_local std::string g_last_error;

int fail(int st, const std::string &msg) {
  g_last_error = msg;
  return st;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
  size_t err, rope, x, h, xg, ssq, qb, kb, vb, attn, act, row_pos, keys, yg, ssq_y, slot, rpos;
  size_t skeys, stickets;   // race keys / tickets of sampled verification, zero between calls
  size_t cfeat, coff, crows, ccount;   // prefix-valid compaction of injected rows (bf16)
  size_t tc_partials, tc_counters, tc_grid_bar;
  int tc_max_tiles;
  size_t att_item_start, att_pps, att_order, att_part_o, att_part_ml, att_tickets;
  int att_bg;
  size_t total;
};

}  // namespace

struct dflash_handle {
  dflash_config cfg;
  std::vector<int32_t> window;
  const void *fc_w, *hidden_norm_g, *final_norm_g, *embed, *lm_head;
  std::vector<const void *> qkv_w, o_w, gate_up_w, down_w, in_norm_g, post_norm_g, q_norm_g,
      k_norm_g;
  Layout L;
  char *ws = nullptr;
  size_t ws_bytes = 0;
  int store;      // ST_F32 / ST_BF16
  bool fuse = true;   // dependent bf16 GEMMs as one cooperative launch
  bool attn_tc = true;  // tcgen05 attention where it applies (else the mma.sync kernel)
  // DFlash 2 candidate selector (dflash_set_selector); K == 0: not set
  struct Selector {
    int K = 0, rank = 0;
    const void *W_h = nullptr, *A = nullptr, *B = nullptr;
    char *ws = nullptr;
    size_t keys = 0, bound = 0, wh = 0, cand = 0;   // offsets into ws
  } sel;
  size_t es;      // element size of the configured dtype
  // optional per-launch event timing
  struct ProfRec {
    const char *name;
    cudaEvent_t a, b;
  };
  bool prof_on = false;
  size_t prof_cap = 0;
  std::vector<cudaEvent_t> ev;
  std::vector<ProfRec> recs;
};

namespace {

Layout plan(const dflash_config &c, size_t es) {
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + std::max<size_t>(bytes, 1), 256);
    return at;
  };
  const size_t M = (size_t)c.max_batch * c.block_size;
  const size_t R = (size_t)c.max_rows;
  const size_t H = c.hidden, D = c.head_dim;
  L.err = take(256);
  L.rope = take(sizeof(float) * 2 * (size_t)c.max_position * (D / 2));
  L.x = take(4 * M * H);
  L.h = take(es * M * H);
  L.xg = take(es * M * H);                       // x * g of the next RMSNorm (GEMM operand)
  L.ssq = take(4 * (H / 128) * M);               // per-128-feature sums of squares of x
  L.qb = take(es * M * c.n_heads * D);
  L.kb = take(es * M * c.n_kv_heads * D);
  L.vb = take(es * M * c.n_kv_heads * D);
  L.attn = take(es * M * c.n_heads * D);
  L.act = take(es * M * c.intermediate);
  L.row_pos = take(4 * M);
  L.keys = take(8 * M);
  L.yg = take(es * R * H);                       // fc output * hidden_norm gain
  L.ssq_y = take(4 * (H / 128) * R);
  L.slot = take(4 * R);
  L.rpos = take(4 * R);
  L.skeys = take(8 * (size_t)c.max_batch);
  L.stickets = take(4 * (size_t)c.max_batch);
  if (es == 2) {
    // the committed rows of a verify block, gathered: up to max_batch *
    // block_size rows of the concatenated target features
    L.cfeat = take(es * std::min(M, R) * (size_t)c.n_sel * c.target_hidden);
    L.coff = take(4 * (size_t)c.max_batch);
    L.crows = take(4 * (size_t)c.max_batch);
    L.ccount = take(4);
  }
  if (es == 2) {
    // tensor-core GEMM scratch: stream-K partial tiles and per-tile tickets
    const int Mb = (int)M, Mr = c.max_rows;
    auto t128 = [](long long n) { return (int)((n + 127) / 128); };
    int mt = 0;
    mt = std::max(mt, gemm_tc_tiles(t128((long long)c.n_heads * D + 2LL * c.n_kv_heads * D), Mb, false));
    mt = std::max(mt, gemm_tc_tiles(t128(H), Mb, false));
    mt = std::max(mt, gemm_tc_tiles(t128(c.intermediate), Mb, true));
    mt = std::max(mt, gemm_tc_tiles(t128(c.vocab), Mb, false));
    mt = std::max(mt, gemm_tc_tiles(t128(H), Mr, false));
    mt = std::max(mt, gemm_tc_tiles(std::min(c.n_layers, kMaxSeg) * t128(2LL * c.n_kv_heads * D), Mr, false));
    L.tc_max_tiles = kMaxPhases * mt;   // tickets of every phase of a fused launch
    L.tc_partials = take(gemm_tc_partials_bytes());
    L.tc_counters = take(4 * (size_t)L.tc_max_tiles);
    L.tc_grid_bar = take(8);
    // attention split scratch
    const size_t R = (size_t)(c.n_heads / c.n_kv_heads) * c.block_size;
    const size_t items = attention_mma_scratch_items(c.max_batch, c.n_kv_heads);
    L.att_bg = c.max_batch * c.n_kv_heads;
    L.att_item_start = take(4 * ((size_t)L.att_bg + 1));
    L.att_pps = take(8);
    L.att_order = take(32 * items);   // the tensor-core kernel's queue: two int4 per item
    L.att_part_o = take(4 * items * R * 128);
    L.att_part_ml = take(8 * items * R);
    L.att_tickets = take(4 * (size_t)L.att_bg);
  }
  L.total = o;
  return L;
}

template <typename P> P *at(dflash_handle *h, size_t off) { return (P *)(h->ws + off); }

int check_cuda(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return DFLASH_OK;
  return fail(DFLASH_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Runs one launch; when profiling is on, brackets it with a pair of events.
template <class F> int timed(dflash_handle *h, const char *name, cudaStream_t s, F &&launch) {
  int idx = -1;
  if (h->prof_on && h->recs.size() < h->prof_cap) {
    idx = (int)h->recs.size();
    h->recs.push_back({name, h->ev[2 * idx], h->ev[2 * idx + 1]});
    cudaEventRecord(h->ev[2 * idx], s);
  }
  const cudaError_t e = launch();
  if (idx >= 0) cudaEventRecord(h->ev[2 * idx + 1], s);
  return check_cuda(e, name);
}

cudaError_t run_gemm(dflash_handle *h, const GemmProblem &P, cudaStream_t s) {
  if (h->store == ST_F32) return launch_gemm_simt(ST_F32, P, s);
  return launch_gemm_tc(P, at<float>(h, h->L.tc_partials), at<int>(h, h->L.tc_counters),
                        h->L.tc_max_tiles, at<unsigned int>(h, h->L.err), s);
}

// Dependent GEMMs of equal row count in one launch (bf16); fp32 runs them one
// after the other on the CUDA cores.
cudaError_t run_program(dflash_handle *h, const GemmProblem *P, int n, cudaStream_t s,
                        const ProgramEmbed *embed = nullptr, const ProgramFinalize *fin = nullptr,
                        const ProgramInject *inject = nullptr, const ProgramNorm *norm = nullptr) {
  if (h->store == ST_F32) {
    for (int i = 0; i < n; ++i) {
      const cudaError_t e = launch_gemm_simt(ST_F32, P[i], s);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  if (!h->fuse) {
    for (int i = 0; i < n; ++i) {
      const cudaError_t e = run_gemm(h, P[i], s);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  return launch_gemm_program(P, n, at<float>(h, h->L.tc_partials), at<int>(h, h->L.tc_counters),
                             h->L.tc_max_tiles, at<unsigned int>(h, h->L.tc_grid_bar),
                             at<unsigned int>(h, h->L.err), s, nullptr, embed, fin, inject, norm);
}

cudaError_t run_attention(dflash_handle *h, const AttnParams &a, cudaStream_t s) {
  if (h->store == ST_F32) return launch_attention_simt(ST_F32, a, s);
  AttnScratch w;
  w.item_start = at<int>(h, h->L.att_item_start);
  w.pps = at<int>(h, h->L.att_pps);
  w.part_o = at<float>(h, h->L.att_part_o);
  w.part_ml = at<float>(h, h->L.att_part_ml);
  w.tickets = at<int>(h, h->L.att_tickets);
  w.order = at<int>(h, h->L.att_order);
  if (h->attn_tc && attention_tc_eligible(a) && !attention_mma_uses_cluster(a))
    return launch_attention_tc(a, w, s);
  return launch_attention_mma(a, w, s);
}

EpiParams epi_base(const dflash_handle *h, int op) {
  EpiParams e;
  std::memset(&e, 0, sizeof(e));
  e.op = op;
  e.n_heads = h->cfg.n_heads;
  e.n_kv_heads = h->cfg.n_kv_heads;
  e.head_dim = h->cfg.head_dim;
  e.eps = h->cfg.rms_eps;
  return e;
}

// The GEMM's A operand is x * g of an RMSNorm whose row scale is applied in
// the epilogue from the per-tile sums of squares `ssq` (row stride ld).
void set_norm_in(const dflash_handle *h, EpiParams &e, const float *ssq, int ld) {
  e.ssq_in = ssq;
  e.ssq_parts = h->cfg.hidden / 128;
  e.ssq_ld = ld;
  e.norm_eps = h->cfg.rms_eps;
  e.inv_h = 1.0f / (float)h->cfg.hidden;
}

GemmProblem problem_1src(const void *A, int64_t lda, int M, int K) {
  GemmProblem P;
  std::memset(&P, 0, sizeof(P));
  P.A.ptr[0] = A;
  P.A.ld = lda;
  P.A.k_per_src = K;
  P.A.n_src = 1;
  P.M = M;
  P.K = K;
  return P;
}

void add_seg(GemmProblem &P, const void *W, int64_t ldw, int N, const EpiParams &e) {
  GemmSeg &s = P.seg[P.nseg++];
  s.W = W;
  s.ldw = ldw;
  s.N = N;
  s.epi = e;
}

// Selector workspace: per-tile top-K keys [ceil(V/128)][max_rows][K], the
// per-row bound slots [K][max_rows], W_h (x*g) [max_rows][rank] fp32 and the merged
// candidates [max_rows][K].
struct SelLayout {
  size_t keys, bound, wh, cand, total;
};
SelLayout sel_layout(const dflash_handle *h, int K, int rank) {
  const dflash_config &c = h->cfg;
  const size_t rows = (size_t)c.max_batch * c.block_size;
  const size_t n_vt = ((size_t)c.vocab + 127) / 128;
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  SelLayout L;
  L.keys = 0;
  L.bound = up(n_vt * rows * K * 8);
  L.wh = L.bound + up(rows * K * 8);
  L.cand = L.wh + up(rows * rank * 4);
  L.total = L.cand + up(rows * K * 8);
  return L;
}

int check_kv(const dflash_handle *h, const dflash_kv *kv) {
  if (!kv) return fail(DFLASH_EINVAL, "kv is NULL");
  if (!kv->k_pages || !kv->v_pages || !kv->page_table || !kv->kv_len)
    return fail(DFLASH_EINVAL, "kv: k_pages, v_pages, page_table and kv_len must be non-NULL");
  if (kv->pages_per_req <= 0 || kv->n_pages <= 0)
    return fail(DFLASH_EINVAL, "kv: pages_per_req and n_pages must be positive");
  for (int l = 0; l < h->cfg.n_layers; ++l)
    if (!kv->k_pages[l] || !kv->v_pages[l])
      return fail(DFLASH_EINVAL, "kv: NULL page pointer for layer " + std::to_string(l));
  if (kv->draft_window < 0) return fail(DFLASH_EINVAL, "kv: negative draft_window");
  if (kv->draft_window > 0 &&
      (int64_t)kv->pages_per_req * h->cfg.page_size < (int64_t)kv->draft_window + h->cfg.page_size)
    return fail(DFLASH_EINVAL, "kv: a draft window of W rows needs a ring of at least "
                               "ceil(W / page_size) + 1 pages per request");
  if (h->cfg.kv_fp8) {
    if (!kv->k_scale || !kv->v_scale) return fail(DFLASH_EINVAL, "kv: FP8 cache without k_scale/v_scale");
    for (int l = 0; l < h->cfg.n_layers; ++l)
      if (!(kv->k_scale[l] > 0.f) || !(kv->v_scale[l] > 0.f) || std::isinf(kv->k_scale[l]) ||
          std::isinf(kv->v_scale[l]))
        return fail(DFLASH_EINVAL, "kv: FP8 scales must be positive and finite");
  }
  return DFLASH_OK;
}
// Capacity of a request's page table in rows (no limit for a draft-window ring).
int64_t kv_capacity(const dflash_handle *h, const dflash_kv *kv) {
  return kv->draft_window > 0 ? (int64_t)INT32_MAX : (int64_t)kv->pages_per_req * h->cfg.page_size;
}

}  // namespace

namespace dflash {
int handle_lm_head(const dflash_handle *h, const void **lm_head, int *hidden, int *vocab,
                   int *dtype) {
  if (!h) return DFLASH_EINVAL;
  *lm_head = h->lm_head;
  *hidden = h->cfg.hidden;
  *vocab = h->cfg.vocab;
  *dtype = h->cfg.dtype;
  return DFLASH_OK;
}
void set_last_error(const char *msg) { g_last_error = msg; }
}  // namespace dflash

extern "C" {

const char *dflash_status_string(int st) {
  switch (st) {
    case DFLASH_OK: return "ok";
    case DFLASH_EINVAL: return "invalid argument";
    case DFLASH_EUNSUPPORTED: return "unsupported shape";
    case DFLASH_ECAPACITY: return "capacity exceeded";
    case DFLASH_ECUDA: return "CUDA error";
    case DFLASH_EDEVICE: return "device-side error flagged";
    case DFLASH_ESTATE: return "no workspace bound";
    default: return "unknown status";
  }
}

const char *dflash_last_error(void) { return g_last_error.c_str(); }

int dflash_create(const dflash_config *cfg, const dflash_weights *w, dflash_handle **out) {
  if (!out) return fail(DFLASH_EINVAL, "out is NULL");
  *out = nullptr;
  if (!cfg || !w) return fail(DFLASH_EINVAL, "cfg and weights must be non-NULL");
  const dflash_config &c = *cfg;
  if (c.dtype != DFLASH_F32 && c.dtype != DFLASH_BF16) return fail(DFLASH_EUNSUPPORTED, "dtype");
  if (c.target_hidden <= 0 || c.n_sel <= 0 || c.hidden <= 0 || c.n_layers <= 0 || c.n_heads <= 0 ||
      c.n_kv_heads <= 0 || c.head_dim <= 0 || c.intermediate <= 0 || c.vocab <= 1 ||
      c.block_size <= 0 || c.max_batch <= 0 || c.max_rows <= 0 || c.max_position <= 0)
    return fail(DFLASH_EINVAL, "every size in the config must be positive");
  if (c.n_sel > kMaxSrc) return fail(DFLASH_EUNSUPPORTED, "n_sel must be <= 8");
  if (c.head_dim != 64 && c.head_dim != 128) return fail(DFLASH_EUNSUPPORTED, "head_dim must be 64 or 128");
  if (c.n_heads % c.n_kv_heads) return fail(DFLASH_EUNSUPPORTED, "n_heads must be a multiple of n_kv_heads");
  if (c.hidden % 128 || c.target_hidden % 128 || c.intermediate % 128 || (c.n_heads * c.head_dim) % 128 ||
      (c.n_kv_heads * c.head_dim) % 64)
    return fail(DFLASH_EUNSUPPORTED, "hidden, target_hidden, intermediate, n_heads*head_dim must be multiples of 128");
  if (c.block_size < 2 || c.block_size > 32) return fail(DFLASH_EUNSUPPORTED, "block_size must be in [2, 32]");
  if ((c.n_heads / c.n_kv_heads) * c.block_size > 128)
    return fail(DFLASH_EUNSUPPORTED, "(n_heads/n_kv_heads)*block_size must be <= 128");
  if (c.page_size != 64) return fail(DFLASH_EUNSUPPORTED, "page_size must be 64");
  if (c.dtype == DFLASH_BF16 && c.head_dim != 128)
    return fail(DFLASH_EUNSUPPORTED, "bf16 configurations need head_dim 128");
  if (c.kv_fp8 != 0 && c.kv_fp8 != 1) return fail(DFLASH_EINVAL, "kv_fp8 must be 0 or 1");
  if (c.kv_fp8 && (c.dtype != DFLASH_BF16 || c.head_dim != 128 || c.block_size > 16))
    return fail(DFLASH_EUNSUPPORTED, "an FP8 KV cache needs bf16, head_dim 128 and block_size <= 16");
  if (c.mask_token_id < 0 || c.mask_token_id >= c.vocab) return fail(DFLASH_EINVAL, "mask_token_id outside the vocabulary");
  if (!(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f)) return fail(DFLASH_EINVAL, "rms_eps >= 0 and rope_theta > 0 required");
  if (c.max_position < c.block_size) return fail(DFLASH_EINVAL, "max_position < block_size");
  if (!c.sliding_window) return fail(DFLASH_EINVAL, "sliding_window array is NULL");
  for (int l = 0; l < c.n_layers; ++l)
    if (c.sliding_window[l] < 0) return fail(DFLASH_EINVAL, "negative sliding_window");
  if (!w->fc_w || !w->hidden_norm_g || !w->final_norm_g || !w->embed || !w->lm_head || !w->qkv_w ||
      !w->o_w || !w->gate_up_w || !w->down_w || !w->in_norm_g || !w->post_norm_g || !w->q_norm_g ||
      !w->k_norm_g)
    return fail(DFLASH_EINVAL, "a weight pointer is NULL");
  for (int l = 0; l < c.n_layers; ++l)
    if (!w->qkv_w[l] || !w->o_w[l] || !w->gate_up_w[l] || !w->down_w[l] || !w->in_norm_g[l] ||
        !w->post_norm_g[l] || !w->q_norm_g[l] || !w->k_norm_g[l])
      return fail(DFLASH_EINVAL, "a per-layer weight pointer is NULL (layer " + std::to_string(l) + ")");
  // the FP8 store runs in the per-head epilogue that reads gains 8 bytes at a time
  if (c.kv_fp8)
    for (int l = 0; l < c.n_layers; ++l)
      if ((uintptr_t)w->k_norm_g[l] % 8 || (uintptr_t)w->q_norm_g[l] % 8)
        return fail(DFLASH_EINVAL, "q/k norm gains must be 8-byte aligned with an FP8 KV cache");

  dflash_handle *h = new dflash_handle();
  h->cfg = c;
  h->window.assign(c.sliding_window, c.sliding_window + c.n_layers);
  h->cfg.sliding_window = h->window.data();
  h->fc_w = w->fc_w;
  h->hidden_norm_g = w->hidden_norm_g;
  h->final_norm_g = w->final_norm_g;
  h->embed = w->embed;
  h->lm_head = w->lm_head;
  const int L = c.n_layers;
  h->qkv_w.assign(w->qkv_w, w->qkv_w + L);
  h->o_w.assign(w->o_w, w->o_w + L);
  h->gate_up_w.assign(w->gate_up_w, w->gate_up_w + L);
  h->down_w.assign(w->down_w, w->down_w + L);
  h->in_norm_g.assign(w->in_norm_g, w->in_norm_g + L);
  h->post_norm_g.assign(w->post_norm_g, w->post_norm_g + L);
  h->q_norm_g.assign(w->q_norm_g, w->q_norm_g + L);
  h->k_norm_g.assign(w->k_norm_g, w->k_norm_g + L);
  h->store = c.dtype == DFLASH_F32 ? ST_F32 : ST_BF16;
  h->es = c.dtype == DFLASH_F32 ? 4 : 2;
  h->L = plan(h->cfg, h->es);
  *out = h;
  g_last_error.clear();
  return DFLASH_OK;
}

void dflash_destroy(dflash_handle *h) {
  if (!h) return;
  for (cudaEvent_t e : h->ev) cudaEventDestroy(e);
  delete h;
}

int dflash_profile_enable(dflash_handle *h, int32_t max_records) {
  if (!h || max_records <= 0) return fail(DFLASH_EINVAL, "handle NULL or max_records <= 0");
  while (h->ev.size() < 2 * (size_t)max_records) {
    cudaEvent_t e;
    if (int st = check_cuda(cudaEventCreate(&e), "cudaEventCreate")) return st;
    h->ev.push_back(e);
  }
  h->prof_cap = (size_t)max_records;
  h->recs.clear();
  h->prof_on = true;
  return DFLASH_OK;
}

int dflash_profile_disable(dflash_handle *h) {
  if (!h) return fail(DFLASH_EINVAL, "handle is NULL");
  h->prof_on = false;
  return DFLASH_OK;
}

int dflash_profile_collect(dflash_handle *h, dflash_profile_entry *out, int32_t cap, int32_t *n) {
  if (!h || !out || !n || cap < 0) return fail(DFLASH_EINVAL, "NULL argument");
  std::vector<dflash_profile_entry> agg;
  for (const auto &r : h->recs) {
    if (int st = check_cuda(cudaEventSynchronize(r.b), "cudaEventSynchronize")) return st;
    float ms = 0.f;
    if (int st = check_cuda(cudaEventElapsedTime(&ms, r.a, r.b), "cudaEventElapsedTime")) return st;
    auto it = std::find_if(agg.begin(), agg.end(),
                           [&](const dflash_profile_entry &e) { return !std::strcmp(e.name, r.name); });
    if (it == agg.end()) {
      dflash_profile_entry e;
      std::memset(&e, 0, sizeof(e));
      std::strncpy(e.name, r.name, sizeof(e.name) - 1);
      agg.push_back(e);
      it = agg.end() - 1;
    }
    it->launches += 1;
    it->total_ms += ms;
  }
  h->recs.clear();
  *n = (int32_t)std::min<size_t>(agg.size(), (size_t)cap);
  for (int i = 0; i < *n; ++i) out[i] = agg[i];
  return DFLASH_OK;
}

int dflash_workspace_size(const dflash_handle *h, size_t *bytes) {
  if (!h || !bytes) return fail(DFLASH_EINVAL, "handle and bytes must be non-NULL");
  *bytes = h->L.total;
  return DFLASH_OK;
}

int dflash_bind_workspace(dflash_handle *h, void *dev_ptr, size_t bytes, dflash_stream_t stream) {
  if (!h || !dev_ptr) return fail(DFLASH_EINVAL, "handle and workspace must be non-NULL");
  if ((uintptr_t)dev_ptr % 256) return fail(DFLASH_EINVAL, "workspace must be 256-byte aligned");
  if (bytes < h->L.total)
    return fail(DFLASH_ECAPACITY, "workspace too small: need " + std::to_string(h->L.total) + " bytes");
  cudaStream_t s = (cudaStream_t)stream;
  h->ws = (char *)dev_ptr;
  h->ws_bytes = bytes;
  int st = check_cuda(cudaMemsetAsync(h->ws + h->L.err, 0, 256, s), "clear error word");
  if (st) return st;
  if (h->L.tc_max_tiles > 0 &&
      (st = check_cuda(cudaMemsetAsync(h->ws + h->L.tc_counters, 0, 4 * (size_t)h->L.tc_max_tiles, s),
                       "clear GEMM tickets")))
    return st;
  if (h->L.tc_max_tiles > 0 &&
      (st = check_cuda(cudaMemsetAsync(h->ws + h->L.tc_grid_bar, 0, 8, s), "clear grid barrier")))
    return st;
  if (h->L.att_bg > 0 &&
      (st = check_cuda(cudaMemsetAsync(h->ws + h->L.att_tickets, 0, 4 * (size_t)h->L.att_bg, s),
                       "clear attention tickets")))
    return st;
  if ((st = check_cuda(cudaMemsetAsync(h->ws + h->L.skeys, 0, 8 * (size_t)h->cfg.max_batch, s),
                       "clear sampled-verification keys")) ||
      (st = check_cuda(cudaMemsetAsync(h->ws + h->L.stickets, 0, 4 * (size_t)h->cfg.max_batch, s),
                       "clear sampled-verification tickets")))
    return st;
  st = check_cuda(launch_rope_table(at<float2>(h, h->L.rope), h->cfg.max_position, h->cfg.head_dim,
                                    h->cfg.rope_theta, s), "rope table");
  if (st) return st;
  return check_cuda(prepare_kernels(), "kernel attributes");
}

int dflash_get_error(dflash_handle *h, dflash_stream_t stream, uint32_t *word) {
  if (!h) return fail(DFLASH_EINVAL, "handle is NULL");
  if (!h->ws) return fail(DFLASH_ESTATE, "no workspace bound");
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t v = 0;
  int st = check_cuda(cudaMemcpyAsync(&v, h->ws + h->L.err, sizeof(v), cudaMemcpyDeviceToHost, s), "read error word");
  if (st) return st;
  st = check_cuda(cudaMemsetAsync(h->ws + h->L.err, 0, sizeof(v), s), "clear error word");
  if (st) return st;
  st = check_cuda(cudaStreamSynchronize(s), "synchronize");
  if (st) return st;
  if (word) *word = v;
  return v ? DFLASH_EDEVICE : DFLASH_OK;
}

int dflash_inject_context(dflash_handle *h, const dflash_kv *kv, int32_t batch, int32_t total_rows,
                          const void *const *target_feats, const int32_t *row_offset,
                          const int32_t *n_rows, dflash_stream_t stream) {
  if (!h) return fail(DFLASH_EINVAL, "handle is NULL");
  if (!h->ws) return fail(DFLASH_ESTATE, "no workspace bound");
  const dflash_config &c = h->cfg;
  if (int st = check_kv(h, kv)) return st;
  if (batch < 0 || total_rows < 0) return fail(DFLASH_EINVAL, "negative batch or total_rows");
  if (batch > c.max_batch) return fail(DFLASH_ECAPACITY, "batch > max_batch");
  if (batch == 0) return DFLASH_OK;
  if (!target_feats || !row_offset || !n_rows)
    return fail(DFLASH_EINVAL, "target_feats, row_offset and n_rows must be non-NULL");
  for (int j = 0; j < c.n_sel; ++j)
    if (!target_feats[j]) return fail(DFLASH_EINVAL, "NULL feature pointer " + std::to_string(j));
  cudaStream_t s = (cudaStream_t)stream;
  unsigned int *err = at<unsigned int>(h, h->L.err);
  const int H = c.hidden, D = c.head_dim;
  const int kvd = c.n_kv_heads * D;
  const int q_rows = c.n_heads * D;
  int *slot = at<int>(h, h->L.slot), *rpos = at<int>(h, h->L.rpos);
  void *yg = h->ws + h->L.yg;
  float *ssq_y = at<float>(h, h->L.ssq_y);
  const float2 *rope = at<const float2>(h, h->L.rope);

  // fused bf16 path: the row map is computed inside the injection launch and,
  // when that launch is the call's last, so is the kv_len update
  const bool fused = h->store == ST_BF16 && h->fuse;
  bool advanced = false;
  // Prefix-valid compaction ("Inside SGLang", Step 7: only the accepted rows
  // of a verify block are written): when the feature rows fit one chunk of
  // the dense [max_batch, block_size] bound, the rows of some request are
  // gathered first and fc and the K/V projections run on them alone; the
  // launches read the row count from the device.  At most 128 rows are one
  // token tile whatever the count, so there it would only add a launch.
  const int64_t gather_cap = std::min<int64_t>(c.max_rows, (int64_t)c.max_batch * c.block_size);
  bool aligned = true;   // the gather copies 16-byte vectors
  for (int j = 0; j < c.n_sel; ++j) aligned = aligned && ((uintptr_t)target_feats[j] & 15) == 0;
  const bool compact =
      fused && aligned && total_rows > 128 && total_rows <= gather_cap && c.n_sel <= kMaxSrc;
  const int32_t *map_off = row_offset, *map_rows = n_rows;
  const int *count = nullptr;
  void *cfeat = h->ws + h->L.cfeat;
  if (compact) {
    FeatPtrs fp;
    std::memset(&fp, 0, sizeof(fp));
    for (int j = 0; j < c.n_sel; ++j) fp.p[j] = target_feats[j];
    int *coff = at<int>(h, h->L.coff), *crows = at<int>(h, h->L.crows);
    int *ccount = at<int>(h, h->L.ccount);
    if (int st = timed(h, "inject_compact", s, [&] {
          return launch_inject_compact(batch, total_rows, fp, c.n_sel, c.target_hidden, row_offset,
                                       n_rows, cfeat, coff, crows, ccount, err, s);
        }))
      return st;
    map_off = coff;
    map_rows = crows;
    count = ccount;
  }
  for (int64_t r0 = 0; r0 < total_rows; r0 += c.max_rows) {
    const int rows = (int)std::min<int64_t>(c.max_rows, total_rows - r0);
    int st = 0;
    if (!fused && (st = timed(h, "inject_prep", s, [&] {
                     return launch_inject_prep(batch, (int)r0, rows, row_offset, n_rows, kv->kv_len,
                                               kv->page_table, kv->pages_per_req, kv->n_pages,
                                               c.page_size, c.max_position, kv->draft_window, slot,
                                               rpos, err, s);
                   })))
      return st;
    // a1 + a2: concat (K-split over the selected layers) + fc; the epilogue
    // writes y * hidden_norm gain and the row sums of squares of y
    GemmProblem prog[2];
    GemmProblem &P = prog[0];
    std::memset(&P, 0, sizeof(P));
    if (compact) {
      // one source: the gathered rows hold the selected layers side by side
      P.A.ptr[0] = cfeat;
      P.A.ld = (int64_t)c.n_sel * c.target_hidden;
      P.A.k_per_src = c.n_sel * c.target_hidden;
      P.A.n_src = 1;
      P.M_dev = count;
    } else {
      for (int j = 0; j < c.n_sel; ++j)
        P.A.ptr[j] = (const char *)target_feats[j] + (size_t)r0 * c.target_hidden * h->es;
      P.A.ld = c.target_hidden;
      P.A.k_per_src = c.target_hidden;
      P.A.n_src = c.n_sel;
    }
    P.M = rows;
    P.K = c.n_sel * c.target_hidden;
    EpiParams e = epi_base(h, EPI_STORE_NORM);
    e.N = H;
    e.ld = H;
    e.out_act = yg;
    e.norm_gain = h->hidden_norm_g;
    e.ssq_out = ssq_y;
    e.ssq_ld = c.max_rows;
    add_seg(P, h->fc_w, P.K, H, e);
    // a3: every layer's K/V projection of hidden_norm(y) + k-norm + RoPE + paged scatter
    auto kv_problem = [&](int l0) {
      GemmProblem Q = problem_1src(yg, H, rows, H);
      Q.M_dev = count;
      for (int l = l0; l < std::min(c.n_layers, l0 + kMaxSeg); ++l) {
        EpiParams k = epi_base(h, EPI_KV_CACHE);
        k.N = 2 * kvd;
        k.k_cache = kv->k_pages[l];
        k.v_cache = kv->v_pages[l];
        k.k_gain = h->k_norm_g[l];
        k.row_pos = rpos;
        k.row_slot = slot;
        k.rope = rope;
        if (c.kv_fp8) {
          k.kv_fp8 = 1;
          k.k_scale = kv->k_scale[l];
          k.v_scale = kv->v_scale[l];
        }
        set_norm_in(h, k, ssq_y, c.max_rows);
        add_seg(Q, (const char *)h->qkv_w[l] + (size_t)q_rows * H * h->es, H, 2 * kvd, k);
      }
      return Q;
    };
    prog[1] = kv_problem(0);
    ProgramInject inj;
    std::memset(&inj, 0, sizeof(inj));
    inj.B = batch;
    inj.row0 = (int)r0;
    inj.rows = rows;
    inj.row_offset = map_off;
    inj.n_rows = map_rows;
    inj.kv_len = kv->kv_len;
    inj.page_table = kv->page_table;
    inj.pages_per_req = kv->pages_per_req;
    inj.n_pages = kv->n_pages;
    inj.page_size = c.page_size;
    inj.max_position = c.max_position;
    inj.row_slot = slot;
    inj.row_pos = rpos;
    inj.total_rows = total_rows;
    inj.draft_window = kv->draft_window;
    inj.advance = r0 + rows >= total_rows && c.n_layers <= kMaxSeg;
    advanced = fused && inj.advance;
    // fc and the first group of layers' K/V in one launch
    if ((st = timed(h, "gemm_inject_program", s,
                    [&] { return run_program(h, prog, 2, s, nullptr, nullptr, fused ? &inj : nullptr); })))
      return st;
    for (int l0 = kMaxSeg; l0 < c.n_layers; l0 += kMaxSeg) {
      GemmProblem Q = kv_problem(l0);
      if ((st = timed(h, "gemm_kv_inject", s, [&] { return run_gemm(h, Q, s); }))) return st;
    }
  }
  if (advanced) return DFLASH_OK;
  return timed(h, "inject_finalize", s, [&] {
    return launch_inject_finalize(batch, total_rows, row_offset, n_rows, kv->kv_len,
                                  (int)kv_capacity(h, kv), err, s);
  });
}

// The draft pass; with `run` the final launch ends in the DFlash 2 candidate
// selector instead of the argmax.
struct SelRun {
  const float *exp_noise;
  int32_t *cand_ids;
  float *q_rows;
};
static int draft_impl(dflash_handle *h, const dflash_kv *kv, int32_t batch,
                      const int32_t *anchor, int32_t *draft_ids, void *hidden_out,
                      dflash_stream_t stream, const SelRun *run) {
  if (!h) return fail(DFLASH_EINVAL, "handle is NULL");
  if (!h->ws) return fail(DFLASH_ESTATE, "no workspace bound");
  const dflash_config &c = h->cfg;
  if (int st = check_kv(h, kv)) return st;
  if (batch < 0) return fail(DFLASH_EINVAL, "negative batch");
  if (batch > c.max_batch) return fail(DFLASH_ECAPACITY, "batch > max_batch");
  if (batch == 0) return DFLASH_OK;
  if (!anchor || !draft_ids) return fail(DFLASH_EINVAL, "anchor and draft_ids must be non-NULL");
  cudaStream_t s = (cudaStream_t)stream;
  unsigned int *err = at<unsigned int>(h, h->L.err);
  const int S = c.block_size, M = batch * S, H = c.hidden, D = c.head_dim;
  const int qd = c.n_heads * D, kvd = c.n_kv_heads * D;
  const int ldq = c.max_batch * S;                 // row stride of the sums of squares
  float *x = at<float>(h, h->L.x);
  void *xg = h->ws + h->L.xg;
  float *ssq = at<float>(h, h->L.ssq);
  void *qb = h->ws + h->L.qb, *kb = h->ws + h->L.kb, *vb = h->ws + h->L.vb;
  void *attn = h->ws + h->L.attn, *act = h->ws + h->L.act;
  int *row_pos = at<int>(h, h->L.row_pos);
  // argmax keys (cleared by the embedding), or with the selector the slots of
  // its per-row bounds, cleared here
  unsigned long long *keys = run ? (unsigned long long *)(h->sel.ws + h->sel.bound)
                                 : at<unsigned long long>(h, h->L.keys);
  if (run && check_cuda(cudaMemsetAsync(keys, 0, (size_t)h->sel.K * ldq * 8, s),
                        "selector bound reset"))
    return DFLASH_ECUDA;
  const float2 *rope = at<const float2>(h, h->L.rope);
  int st;

  // fused bf16 path: the embedding runs as the first phase of the layer-0
  // QKV launch, the argmax ids are written by the last CTA of the final launch
  const bool fused = h->store == ST_BF16 && h->fuse;
  // a4: block embedding [anchor, MASK x (S-1)] at positions kv_len + j, with the
  // first layer's input RMSNorm deferred into its QKV GEMM
  if (!fused && (st = timed(h, "embed", s, [&] {
                   return launch_embed(h->store, h->embed, anchor, kv->kv_len, batch, S, H,
                                       c.vocab, c.mask_token_id, c.max_position, x,
                                       h->in_norm_g[0], xg, ssq, ldq, row_pos, keys, err, s);
                 })))
    return st;
  // a5 of layer l: RMSNorm + QKV GEMM + q/k-norm + RoPE
  auto qkv_problem = [&](int l) {
    GemmProblem P = problem_1src(xg, H, M, H);
    EpiParams e = epi_base(h, EPI_QKV);
    e.N = qd + 2 * kvd;
    e.q_out = qb;
    e.k_out = kb;
    e.v_out = vb;
    e.q_gain = h->q_norm_g[l];
    e.k_gain = h->k_norm_g[l];
    e.row_pos = row_pos;
    e.rope = rope;
    set_norm_in(h, e, ssq, ldq);
    add_seg(P, h->qkv_w[l], H, qd + 2 * kvd, e);
    return P;
  };
  {
    GemmProblem P = qkv_problem(0);
    if (fused) {
      ProgramEmbed em;
      em.table = h->embed;
      em.anchor = anchor;
      em.kv_len = kv->kv_len;
      em.M = M;
      em.S = S;
      em.H = H;
      em.vocab = c.vocab;
      em.mask_id = c.mask_token_id;
      em.max_position = c.max_position;
      em.x = x;
      em.gain = h->in_norm_g[0];
      em.xg = xg;
      em.ssq = ssq;
      em.ssq_ld = ldq;
      em.row_pos = row_pos;
      em.keys = keys;
      if ((st = timed(h, "gemm_embed_qkv_program", s, [&] { return run_program(h, &P, 1, s, &em); })))
        return st;
    } else if ((st = timed(h, "gemm_qkv", s, [&] { return run_gemm(h, P, s); }))) {
      return st;
    }
  }
  for (int l = 0; l < c.n_layers; ++l) {
    // a6: non-causal block attention over [context ; block]
    AttnParams a;
    std::memset(&a, 0, sizeof(a));
    a.q = qb;
    a.kb = kb;
    a.vb = vb;
    a.k_cache = kv->k_pages[l];
    a.v_cache = kv->v_pages[l];
    a.page_table = kv->page_table;
    a.kv_len = kv->kv_len;
    a.out = attn;
    a.B = batch;
    a.S = S;
    a.n_heads = c.n_heads;
    a.n_kv_heads = c.n_kv_heads;
    a.head_dim = D;
    a.page_size = c.page_size;
    a.pages_per_req = kv->pages_per_req;
    a.n_pages = kv->n_pages;
    a.window = h->window[l];
    a.scale = 1.0f / sqrtf((float)D);
    a.err = err;
    a.draft_window = kv->draft_window;
    if (c.kv_fp8) {
      a.fp8 = 1;
      a.k_scale = kv->k_scale[l];
      a.v_scale = kv->v_scale[l];
    }
    if ((st = timed(h, "attention", s, [&] { return run_attention(h, a, s); }))) return st;
    // One launch for the rest of the layer and the start of the next:
    // a7 O-proj + residual (+ deferred post-attention norm), a8 gate/up with
    // SwiGLU, down + residual (+ deferred next norm), then the next layer's
    // QKV (a5) or, after the last layer, the lm_head with argmax (a9).
    GemmProblem prog[4];
    prog[0] = problem_1src(attn, qd, M, qd);
    EpiParams eo = epi_base(h, EPI_RESID_NORM);
    eo.N = H;
    eo.ld = H;
    eo.out_f32 = x;
    eo.out_act = xg;
    eo.norm_gain = h->post_norm_g[l];
    eo.ssq_out = ssq;
    eo.ssq_ld = ldq;
    add_seg(prog[0], h->o_w[l], qd, H, eo);
    prog[1] = problem_1src(xg, H, M, H);
    EpiParams eg = epi_base(h, EPI_SWIGLU);
    eg.N = 2 * c.intermediate;
    eg.ld = c.intermediate;
    eg.out_act = act;
    set_norm_in(h, eg, ssq, ldq);
    add_seg(prog[1], h->gate_up_w[l], H, 2 * c.intermediate, eg);
    prog[2] = problem_1src(act, c.intermediate, M, c.intermediate);
    EpiParams ed = epi_base(h, EPI_RESID_NORM);
    ed.N = H;
    ed.ld = H;
    ed.out_f32 = x;
    ed.out_act = xg;
    ed.norm_gain = l + 1 < c.n_layers ? h->in_norm_g[l + 1] : h->final_norm_g;
    ed.ssq_out = ssq;
    ed.ssq_ld = ldq;
    add_seg(prog[2], h->down_w[l], c.intermediate, H, ed);
    if (l + 1 < c.n_layers) {
      prog[3] = qkv_problem(l + 1);
      if ((st = timed(h, "gemm_layer_program", s, [&] { return run_program(h, prog, 4, s); })))
        return st;
    } else {
      // a9: final norm, lm_head + argmax (logits never stored).  The lm_head
      // reads the final-normed rows rounded to the store type -- the same
      // values hidden_out receives -- so the drafted ids are exactly the
      // argmax of the hidden states the caller sees.
      prog[3] = problem_1src(xg, H, M, H);
      EpiParams ea = epi_base(h, run ? EPI_TOPK : EPI_ARGMAX);
      ea.N = c.vocab;
      ea.argmax_keys = keys;
      if (run) {
        // DFlash 2: every row's K best tokens per vocabulary tile, and W_h of
        // the same operand as a second segment of the launch
        ea.topk_keys = (unsigned long long *)(h->sel.ws + h->sel.keys);
        ea.topk_bound = keys;
        ea.topk = h->sel.K;
        ea.topk_ld = ldq;
      }
      add_seg(prog[3], h->lm_head, H, c.vocab, ea);
      if (run) {
        EpiParams ew = epi_base(h, EPI_STORE_F32);
        ew.N = h->sel.rank;
        ew.ld = h->sel.rank;
        ew.out_f32 = (float *)(h->sel.ws + h->sel.wh);
        add_seg(prog[3], h->sel.W_h, H, h->sel.rank, ew);
      }
      ProgramFinalize fin;
      fin.keys = keys;
      fin.anchor = anchor;
      fin.M = M;
      fin.S = S;
      fin.draft_ids = draft_ids;
      if (fused && H % 256 == 0) {
        // O, gate/up, down, the final norm (a GEMM-free phase) and the lm_head
        ProgramNorm nm;
        nm.x = x;
        nm.ssq = ssq;
        nm.ssq_ld = ldq;
        nm.gain = h->final_norm_g;
        nm.out = xg;
        nm.out2 = hidden_out;
        nm.M = M;
        nm.H = H;
        nm.eps = c.rms_eps;
        if ((st = timed(h, "gemm_last_program", s, [&] {
               return run_program(h, prog, 4, s, nullptr, run ? nullptr : &fin, nullptr, &nm);
             })))
          return st;
      } else {
        if ((st = timed(h, "gemm_last_layer_program", s, [&] { return run_program(h, prog, 3, s); })))
          return st;
        if ((st = timed(h, "rmsnorm_final", s, [&] {
               return launch_rmsnorm(1, h->store, x, h->final_norm_g, M, H, c.rms_eps, xg,
                                     hidden_out, s);
             })))
          return st;
        if ((st = timed(h, "gemm_lm_head", s, [&] {
               return fused ? run_program(h, &prog[3], 1, s, nullptr, run ? nullptr : &fin)
                            : run_gemm(h, prog[3], s);
             })))
          return st;
      }
    }
  }
  if (run) {
    SelectorParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.topk_keys = (const unsigned long long *)(h->sel.ws + h->sel.keys);
    sp.n_vt = (c.vocab + 127) / 128;
    sp.topk_ld = ldq;
    sp.cand_keys = (unsigned long long *)(h->sel.ws + h->sel.cand);
    sp.wh = (const float *)(h->sel.ws + h->sel.wh);
    sp.ssq = nullptr;   // the lm_head operand is already the normalised hidden state
    sp.ssq_ld = ldq;
    sp.H = H;
    sp.eps = c.rms_eps;
    sp.A = h->sel.A;
    sp.Bf = h->sel.B;
    sp.store = h->store;
    sp.anchor = anchor;
    sp.exp_noise = run->exp_noise;
    sp.draft_ids = draft_ids;
    sp.cand_ids = run->cand_ids;
    sp.q_rows = run->q_rows;
    sp.B = batch;
    sp.S = S;
    sp.K = h->sel.K;
    sp.rank = h->sel.rank;
    sp.vocab = c.vocab;
    sp.err = err;
    return timed(h, "selector_walk", s, [&] { return launch_selector_walk(sp, s); });
  }
  if (fused && !run) return DFLASH_OK;   // the ids came with the last launch
  return timed(h, "argmax_finalize", s,
               [&] { return launch_argmax_finalize(keys, anchor, batch, S, draft_ids, s); });
}

int dflash_draft_block(dflash_handle *h, const dflash_kv *kv, int32_t batch, const int32_t *anchor,
                       int32_t *draft_ids, void *hidden_out, dflash_stream_t stream) {
  return draft_impl(h, kv, batch, anchor, draft_ids, hidden_out, stream, nullptr);
}

int dflash_selector_workspace_size(const dflash_handle *h, int32_t K, int32_t rank,
                                   size_t *bytes) {
  if (!h || !bytes) return fail(DFLASH_EINVAL, "handle and bytes must be non-NULL");
  if (K < 1 || K > kSelMaxK || K > h->cfg.vocab)
    return fail(DFLASH_EUNSUPPORTED, "selector: K must be in [1, 8] and at most vocab");
  if (rank < 1 || rank > kSelMaxRank) return fail(DFLASH_EUNSUPPORTED, "selector: rank must be in [1, 256]");
  *bytes = sel_layout(h, K, rank).total;
  return DFLASH_OK;
}

int dflash_set_selector(dflash_handle *h, const dflash_selector *sel, void *workspace,
                        size_t bytes) {
  if (!h) return fail(DFLASH_EINVAL, "handle is NULL");
  if (!sel) {
    h->sel = dflash_handle::Selector();
    return DFLASH_OK;
  }
  size_t need = 0;
  if (int st = dflash_selector_workspace_size(h, sel->K, sel->rank, &need)) return st;
  if (!sel->W_h || !sel->A || !sel->B)
    return fail(DFLASH_EINVAL, "selector: W_h, A and B must be non-NULL");
  if (!workspace || bytes < need) return fail(DFLASH_ECAPACITY, "selector workspace too small");
  if ((uintptr_t)workspace & 255) return fail(DFLASH_EINVAL, "selector workspace must be 256-byte aligned");
  if (h->cfg.block_size - 1 > 32) return fail(DFLASH_EUNSUPPORTED, "selector: block_size above 33");
  if (h->store == ST_BF16 && (((uintptr_t)sel->W_h & 15) || (h->cfg.hidden * 2) % 16))
    return fail(DFLASH_EINVAL, "selector: W_h must be 16-byte aligned");
  const SelLayout L = sel_layout(h, sel->K, sel->rank);
  h->sel.K = sel->K;
  h->sel.rank = sel->rank;
  h->sel.W_h = sel->W_h;
  h->sel.A = sel->A;
  h->sel.B = sel->B;
  h->sel.ws = (char *)workspace;
  h->sel.keys = L.keys;
  h->sel.bound = L.bound;
  h->sel.wh = L.wh;
  h->sel.cand = L.cand;
  return DFLASH_OK;
}

int dflash_draft_block_selector(dflash_handle *h, const dflash_kv *kv, int32_t batch,
                                const int32_t *anchor, const float *exp_noise,
                                int32_t *draft_ids, int32_t *cand_ids, float *q_rows,
                                dflash_stream_t stream) {
  if (!h) return fail(DFLASH_EINVAL, "handle is NULL");
  if (h->sel.K == 0) return fail(DFLASH_ESTATE, "no selector set (dflash_set_selector)");
  SelRun run = {exp_noise, cand_ids, q_rows};
  return draft_impl(h, kv, batch, anchor, draft_ids, nullptr, stream, &run);
}

int dflash_accept_commit_sampled(dflash_handle *h, int32_t batch, const int32_t *draft_ids,
                                 const float *probs, const float *accept_u, const float *exp_noise,
                                 int32_t *seq_len, int32_t *accept_len, int32_t *commit_len,
                                 int32_t *bonus, int32_t *out_tokens, int32_t *output_ids,
                                 int32_t out_stride, dflash_stream_t stream) {
  if (!h) return fail(DFLASH_EINVAL, "handle is NULL");
  if (!h->ws) return fail(DFLASH_ESTATE, "no workspace bound");
  if (batch < 0) return fail(DFLASH_EINVAL, "negative batch");
  if (batch > h->cfg.max_batch) return fail(DFLASH_ECAPACITY, "batch > max_batch");
  if (batch == 0) return DFLASH_OK;
  if (!draft_ids || !probs || !accept_u || !exp_noise || !seq_len || !accept_len || !commit_len ||
      !bonus || !out_tokens)
    return fail(DFLASH_EINVAL, "a required pointer is NULL");
  if (output_ids && out_stride <= 0) return fail(DFLASH_EINVAL, "out_stride must be positive");
  cudaStream_t s = (cudaStream_t)stream;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return timed(h, "accept_sampled", s, [&] {
    return launch_accept_sampled(batch, h->cfg.block_size, h->cfg.vocab, draft_ids, probs, accept_u,
                                 exp_noise, at<unsigned long long>(h, h->L.skeys),
                                 at<int>(h, h->L.stickets), seq_len,
                                 accept_len, commit_len, bonus, out_tokens, output_ids, out_stride,
                                 at<unsigned int>(h, h->L.err), s, sms > 0 ? sms : 1);
  });
}

int dflash_accept_commit_sampled_q(dflash_handle *h, int32_t batch, const int32_t *draft_ids,
                                   const float *probs, int32_t K, const int32_t *cand_ids,
                                   const float *q_rows, const float *accept_u,
                                   const float *exp_noise, int32_t *seq_len, int32_t *accept_len,
                                   int32_t *commit_len, int32_t *bonus, int32_t *out_tokens,
                                   int32_t *output_ids, int32_t out_stride,
                                   dflash_stream_t stream) {
  if (!h) return fail(DFLASH_EINVAL, "handle is NULL");
  if (!h->ws) return fail(DFLASH_ESTATE, "no workspace bound");
  if (batch < 0) return fail(DFLASH_EINVAL, "negative batch");
  if (batch > h->cfg.max_batch) return fail(DFLASH_ECAPACITY, "batch > max_batch");
  if (batch == 0) return DFLASH_OK;
  if (K < 1 || K > kSelMaxK) return fail(DFLASH_EUNSUPPORTED, "K must be in [1, 8]");
  if (!draft_ids || !probs || !cand_ids || !q_rows || !accept_u || !exp_noise || !seq_len ||
      !accept_len || !commit_len || !bonus || !out_tokens)
    return fail(DFLASH_EINVAL, "a required pointer is NULL");
  if (output_ids && out_stride <= 0) return fail(DFLASH_EINVAL, "out_stride must be positive");
  cudaStream_t s = (cudaStream_t)stream;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return timed(h, "accept_sampled_q", s, [&] {
    return launch_accept_sampled(batch, h->cfg.block_size, h->cfg.vocab, draft_ids, probs, accept_u,
                                 exp_noise, at<unsigned long long>(h, h->L.skeys),
                                 at<int>(h, h->L.stickets), seq_len, accept_len, commit_len, bonus,
                                 out_tokens, output_ids, out_stride, at<unsigned int>(h, h->L.err), s,
                                 sms > 0 ? sms : 1, cand_ids, q_rows, K);
  });
}

int dflash_test_set_fusion(dflash_handle *h, int32_t on) {
  if (!h) return fail(DFLASH_EINVAL, "handle is NULL");
  h->fuse = on != 0;
  return DFLASH_OK;
}

int dflash_test_set_attention(dflash_handle *h, int32_t kernel) {
  if (!h) return fail(DFLASH_EINVAL, "handle is NULL");
  if (kernel != 0 && kernel != 1) return fail(DFLASH_EINVAL, "attention kernel must be 0 or 1");
  h->attn_tc = kernel == 0;
  return DFLASH_OK;
}

int dflash_test_set_head_pairs(int32_t on) {
  if (on != 0 && on != 1) return fail(DFLASH_EINVAL, "head pairs must be 0 or 1");
  gemm_tc_set_head_pairs(on == 1);
  return DFLASH_OK;
}

int dflash_accept_commit(dflash_handle *h, int32_t batch, const int32_t *draft_ids,
                         const int32_t *posterior, int32_t *seq_len, int32_t *accept_len,
                         int32_t *commit_len, int32_t *bonus, int32_t *out_tokens,
                         int32_t *output_ids, int32_t out_stride, dflash_stream_t stream) {
  if (!h) return fail(DFLASH_EINVAL, "handle is NULL");
  if (!h->ws) return fail(DFLASH_ESTATE, "no workspace bound");
  if (batch < 0) return fail(DFLASH_EINVAL, "negative batch");
  if (batch > h->cfg.max_batch) return fail(DFLASH_ECAPACITY, "batch > max_batch");
  if (batch == 0) return DFLASH_OK;
  if (!draft_ids || !posterior || !seq_len || !accept_len || !commit_len || !bonus || !out_tokens)
    return fail(DFLASH_EINVAL, "a required pointer is NULL");
  if (output_ids && out_stride <= 0) return fail(DFLASH_EINVAL, "out_stride must be positive");
  cudaStream_t s = (cudaStream_t)stream;
  return timed(h, "accept", s, [&] {
    return launch_accept(batch, h->cfg.block_size, h->cfg.vocab, draft_ids, posterior, seq_len,
                         accept_len, commit_len, bonus, out_tokens, output_ids, out_stride,
                         at<unsigned int>(h, h->L.err), s);
  });
}

}  // extern "C"
