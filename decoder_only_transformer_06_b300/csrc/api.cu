// C ABI of the GPT-2 training-step library: model state, memory plan, host
// init, and the orchestration of one forward / backward / optimizer step.
#include "gpt2.h"
#include "common.cuh"

#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <mutex>
#include <thread>
#include <vector>

#define GPT2_VERSION "gpt2-b300 0.1.0 (sm_103a)"
static const double PI_D = 3.14159265358979323846;

namespace {

struct TensorRec {
    std::string name;
    int ndim;
    int64_t shape[2];
    int64_t offset;   // elements into the arenas
    int64_t numel;
    bool decays;
};

struct LayerActs {
    float* x_in;      // residual stream entering the layer (fp32 [M,C])
    float* x_mid;     // after the attention branch
    void* u1;         // ln_1 output (act [M,C])
    float* mu1;
    float* rs1;
    void* qkv;        // act [M,3C]
    void* att;        // attention output, heads side by side (act [M,C])
    float* lse;       // [B,H,T]
    void* u2;
    float* mu2;
    float* rs2;
    void* hpre;       // gelu'(fc output), saved for the backward (act [M,4C])
    void* hgel;       // after GELU
};

// canonical per-layer tensor order (after wte, wpe)
enum { T_LN1G, T_LN1B, T_ATTW, T_ATTB, T_APW, T_APB, T_LN2G, T_LN2B, T_FCW, T_FCB, T_MPW, T_MPB,
       T_PER_LAYER };

std::string g_create_error = "no error";

}  // namespace

struct gpt2_model {
    gpt2_config cfg{};
    int L = 0, H = 0, C = 0, hs = 0, V = 0, Vp = 0, T = 0, B = 0, M = 0, accum = 1;
    bool use_bf16 = false;
    size_t act_bytes = 4;
    cudaStream_t stream = nullptr;
    // Weight-gradient work of the backward (dW GEMMs, their split-K reduce,
    // bias column sums) runs here, forked from and joined back to `stream`
    // by events, so that it fills the SMs the main chain leaves idle.
    cudaStream_t side = nullptr;
    std::vector<cudaEvent_t> xev;
    int xev_next = 0;
    // AdamW also runs on the side stream, in groups in the order the next
    // forward reads the parameters (embeddings, layer 0..L-1, final
    // LayerNorm); upd_ev[g] marks group g done. While upd_pending, the next
    // forward waits for each group just before it uses it, and every other
    // entry point first joins the side stream.
    std::vector<cudaEvent_t> upd_ev;
    bool upd_pending = false;
    std::vector<std::vector<std::pair<int64_t, int64_t>>> upd_runs;   // [group] arena [begin, end)

    std::vector<TensorRec> tensors;
    int64_t n_arena = 0, decay_end = 0;
    float* params = nullptr;
    float* grads = nullptr;
    float* adam_m = nullptr;
    float* adam_v = nullptr;
    bf16* pbf = nullptr;        // bf16 copy of [0, decay_end)

    std::vector<LayerActs> la;
    float* x_final = nullptr;
    void* uf = nullptr;
    float* muf = nullptr;
    float* rsf = nullptr;
    void* logits = nullptr;
    float* row_loss = nullptr;
    float* last_logits = nullptr;   // fp32 [B, Vp]: the head on one position per sequence
    // Key/value cache of generation: the qkv buffer of every layer holds the
    // keys and values of positions 0..kv_len-1 of the current generation
    // context (set by gpt2_forward_last and gpt2_decode_step; any training
    // forward or parameter change resets it to 0).
    int kv_len = 0;
    void* dec_ws = nullptr;         // row buffers of gpt2_decode_step (allocated on first use)

    float* dres = nullptr;
    void* dres_act = nullptr;
    void* du = nullptr;
    void* dqkv = nullptr;
    void* datt = nullptr;
    void* yproj = nullptr;   // output of a residual-branch projection (act [M,C]), forward only
    void* dh = nullptr;
    float* Dbuf = nullptr;
    float* ln_partial = nullptr;
    float* cs_partial = nullptr;
    float* fc_cs_part = nullptr;   // bf16: [ceil(M/32), 4C] column sums of dh from the c_proj dX GEMM
    float* splitk_ws = nullptr;
    size_t splitk_ws_floats = 0;
    void* emb_ws = nullptr;
    double* norm_partial = nullptr;
    int norm_parts = 0;
    DevState* st = nullptr;

    const int32_t* last_tok = nullptr;
    bool have_targets = false;

    // profiling (see gpt2_profile)
    struct SiteAcc {
        const char* name;
        int64_t calls, kernels;
        double ms, flops, bytes;
    };
    bool prof_on = false;
    std::vector<cudaEvent_t> prof_ev;
    int prof_next = 0;
    std::vector<std::pair<int, int>> prof_pending;   // (site, event index)
    std::vector<SiteAcc> sites;
    std::string err = "no error";
    std::vector<void*> allocs;
    int allocs_tried = 0;       // device allocations attempted (fault injection)

    // --- helpers
    float* P(int i) const { return params + tensors[i].offset; }
    float* G(int i) const { return grads + tensors[i].offset; }
    // GEMM view of a weight: bf16 copy in bf16 mode, fp32 master otherwise
    const void* W(int i) const {
        return use_bf16 ? (const void*)(pbf + tensors[i].offset) : (const void*)(params + tensors[i].offset);
    }
    int lt(int l, int k) const { return 2 + l * T_PER_LAYER + k; }
    int lnf_g() const { return 2 + L * T_PER_LAYER; }
};

static int fail(gpt2_model* m, int code, const std::string& msg) {
    if (m) m->err = msg;
    else g_create_error = msg;
    return code;
}
static int fail_cuda(gpt2_model* m, const char* what, cudaError_t e) {
    return fail(m, GPT2_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}
#define CK(m, expr)                                                 \
    do {                                                            \
        cudaError_t e__ = (expr);                                   \
        if (e__ != cudaSuccess) return fail_cuda((m), #expr, e__);  \
    } while (0)

// ------------------------------------------------------------------ host init
// SplitMix64 (Steele, Lea & Flood 2014): output of a generator advanced once
// from `state`.
static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
static const uint64_t GOLDEN = 0x9E3779B97F4A7C15ull;

// Standard normal for element i of tensor k: state = seed ^ (k*2^40 + i);
// r1, r2 the first two SplitMix64 outputs; u1 = ((r1>>11)+1)*2^-53 in (0,1],
// u2 = (r2>>11)*2^-53 in [0,1); z = sqrt(-2 ln u1) cos(2 pi u2) (Box-Muller).
static inline double init_normal(uint64_t seed, int k, uint64_t i) {
    uint64_t state = seed ^ ((uint64_t)k * (1ull << 40) + i);
    uint64_t r1 = mix64(state + GOLDEN);
    uint64_t r2 = mix64(state + 2 * GOLDEN);
    double u1 = ((double)(r1 >> 11) + 1.0) * (1.0 / 9007199254740992.0);
    double u2 = (double)(r2 >> 11) * (1.0 / 9007199254740992.0);
    return std::sqrt(-2.0 * std::log(u1)) * std::cos(2.0 * PI_D * u2);
}

struct Plan {
    std::vector<TensorRec> t;
    int64_t n_arena = 0, decay_end = 0;
};

static int validate_cfg(const gpt2_config* c, std::string& why) {
    if (!c) { why = "config is NULL"; return GPT2_EINVAL; }
    if (c->n_layer <= 0 || c->n_head <= 0 || c->d_model <= 0 || c->vocab_size <= 0 ||
        c->block_size <= 0 || c->batch_size <= 0 || c->seq_len <= 0) {
        why = "every size must be positive"; return GPT2_EINVAL;
    }
    if (c->d_model % c->n_head) { why = "d_model must be a multiple of n_head"; return GPT2_EINVAL; }
    if (c->seq_len > c->block_size) { why = "seq_len exceeds block_size"; return GPT2_EINVAL; }
    if (c->precision != GPT2_FP32 && c->precision != GPT2_BF16) {
        why = "precision must be GPT2_FP32 or GPT2_BF16"; return GPT2_EINVAL;
    }
    int Vp = c->padded_vocab ? c->padded_vocab : ((c->vocab_size + 127) / 128) * 128;
    if (Vp < c->vocab_size || Vp % 64) {
        why = "padded_vocab must be >= vocab_size and a multiple of 64"; return GPT2_EINVAL;
    }
    if (c->d_model % 32) { why = "d_model must be a multiple of 32"; return GPT2_EINVAL; }
    if (c->d_model > 2048) { why = "d_model above 2048 is not supported"; return GPT2_EINVAL; }
    int hs = c->d_model / c->n_head;
    if (hs > 128) { why = "head size above 128 is not supported"; return GPT2_EINVAL; }
    int64_t M = (int64_t)c->batch_size * c->seq_len;
    if (M > 32768) { why = "batch_size*seq_len above 32768 is not supported"; return GPT2_EINVAL; }
    if ((uint64_t)Vp * (uint64_t)M >= (1ull << 32)) {
        why = "padded_vocab*batch_size*seq_len must be below 2^32"; return GPT2_EINVAL;
    }
    if (c->precision == GPT2_BF16) {
        if (hs != 64) { why = "bf16 mode needs head size 64"; return GPT2_EINVAL; }
        if (c->d_model % 64) { why = "bf16 mode needs d_model % 64 == 0"; return GPT2_EINVAL; }
    }
    if (c->grad_accum_steps < 0) { why = "grad_accum_steps must be >= 0"; return GPT2_EINVAL; }
    return GPT2_OK;
}

// Canonical tensor list; the arena keeps every 2-D tensor first (so AdamW's
// decay mask is one comparison) and aligns each tensor to 64 elements.
static Plan make_plan(const gpt2_config* c) {
    Plan p;
    const int C = c->d_model, L = c->n_layer;
    const int Vp = c->padded_vocab ? c->padded_vocab : ((c->vocab_size + 127) / 128) * 128;
    auto add = [&](const std::string& n, int64_t a, int64_t b) {
        TensorRec r;
        r.name = n;
        r.ndim = b ? 2 : 1;
        r.shape[0] = a;
        r.shape[1] = b;
        r.numel = b ? a * b : a;
        r.decays = b != 0;
        r.offset = -1;
        p.t.push_back(r);
    };
    add("wte", Vp, C);
    add("wpe", c->block_size, C);
    for (int l = 0; l < L; l++) {
        std::string h = "h" + std::to_string(l) + ".";
        add(h + "ln1.g", C, 0);
        add(h + "ln1.b", C, 0);
        add(h + "attn.W", 3 * C, C);
        add(h + "attn.b", 3 * C, 0);
        add(h + "attn_proj.W", C, C);
        add(h + "attn_proj.b", C, 0);
        add(h + "ln2.g", C, 0);
        add(h + "ln2.b", C, 0);
        add(h + "fc.W", 4 * C, C);
        add(h + "fc.b", 4 * C, 0);
        add(h + "mlp_proj.W", C, 4 * C);
        add(h + "mlp_proj.b", C, 0);
    }
    add("lnf.g", C, 0);
    add("lnf.b", C, 0);
    int64_t off = 0;
    for (int pass = 0; pass < 2; pass++) {
        for (auto& r : p.t) {
            if (r.decays != (pass == 0)) continue;
            r.offset = off;
            off += (r.numel + 63) / 64 * 64;
        }
        if (pass == 0) p.decay_end = off;
    }
    p.n_arena = off;
    return p;
}

static void host_init_tensor(const gpt2_config* c, const TensorRec& r, int k, uint64_t seed,
                             float* dst) {
    const bool gain = r.name.size() >= 2 && r.name.compare(r.name.size() - 2, 2, ".g") == 0;
    const bool is_resid = r.name.find("attn_proj.W") != std::string::npos ||
                          r.name.find("mlp_proj.W") != std::string::npos;
    if (r.ndim == 1) {
        for (int64_t i = 0; i < r.numel; i++) dst[i] = gain ? 1.0f : 0.0f;
        return;
    }
    const double std_ = is_resid ? 0.02 / std::sqrt(2.0 * c->n_layer) : 0.02;
    const int nthreads = r.numel > (1 << 20) ? 8 : 1;
    std::vector<std::thread> th;
    for (int w = 0; w < nthreads; w++) {
        th.emplace_back([&, w]() {
            int64_t a = r.numel * w / nthreads, b = r.numel * (w + 1) / nthreads;
            for (int64_t i = a; i < b; i++) dst[i] = (float)(std_ * init_normal(seed, k, (uint64_t)i));
        });
    }
    for (auto& t : th) t.join();
}

// ------------------------------------------------------------------ create
// Fault injection for tests, on the host only: with GPT2_FAIL_ALLOC_AT=n in
// the environment, the n-th device allocation of a gpt2_create (counting from
// 0) fails as if the device had run out of memory, before any cudaMalloc.
static int alloc_dev(gpt2_model* m, void** p, size_t bytes) {
    if (bytes == 0) bytes = 16;
    const int attempt = m->allocs_tried++;
    if (const char* env = std::getenv("GPT2_FAIL_ALLOC_AT")) {
        char* end = nullptr;
        const long at = std::strtol(env, &end, 10);
        if (end != env && at == attempt)
            return fail(m, GPT2_ENOMEM, "injected allocation failure at allocation " +
                                            std::to_string(attempt) + " (GPT2_FAIL_ALLOC_AT)");
    }
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(m, GPT2_ENOMEM, "cudaMalloc of " + std::to_string(bytes) + " bytes failed: " +
                                        cudaGetErrorString(e));
    }
    m->allocs.push_back(*p);
    return GPT2_OK;
}
#define ALLOC(m, ptr, bytes)                                              \
    do {                                                                  \
        void* p__ = nullptr;                                              \
        int r__ = alloc_dev((m), &p__, (bytes));                          \
        if (r__) return r__;                                              \
        (ptr) = (decltype(ptr))p__;                                       \
    } while (0)

static int create_impl(gpt2_model* m, const gpt2_config* cfg, uint64_t seed) {
    m->cfg = *cfg;
    m->L = cfg->n_layer;
    m->H = cfg->n_head;
    m->C = cfg->d_model;
    m->hs = m->C / m->H;
    m->V = cfg->vocab_size;
    m->Vp = cfg->padded_vocab ? cfg->padded_vocab : ((m->V + 127) / 128) * 128;
    m->T = cfg->seq_len;
    m->B = cfg->batch_size;
    m->M = m->B * m->T;
    m->accum = cfg->grad_accum_steps > 0 ? cfg->grad_accum_steps : 1;
    m->use_bf16 = cfg->precision == GPT2_BF16;
    m->act_bytes = m->use_bf16 ? 2 : 4;
    Plan p = make_plan(cfg);
    m->tensors = p.t;
    m->n_arena = p.n_arena;
    m->decay_end = p.decay_end;
    {
        // AdamW groups in the order the forward reads them: 0 = wte, wpe;
        // 1 + l = layer l; L + 1 = final LayerNorm. Each tensor's run extends to
        // the next tensor's offset (covering its alignment padding); adjacent
        // runs of one group merge.
        const int G = m->L + 2;
        m->upd_runs.assign(G, {});
        std::vector<int> order(m->tensors.size());
        for (size_t i = 0; i < order.size(); i++) order[i] = (int)i;
        std::sort(order.begin(), order.end(),
                  [&](int a, int b) { return m->tensors[a].offset < m->tensors[b].offset; });
        for (size_t k = 0; k < order.size(); k++) {
            const int i = order[k];
            const int g = i < 2 ? 0 : (i < 2 + m->L * T_PER_LAYER ? 1 + (i - 2) / T_PER_LAYER : m->L + 1);
            const int64_t b = m->tensors[i].offset;
            const int64_t e = k + 1 < order.size() ? m->tensors[order[k + 1]].offset : m->n_arena;
            auto& runs = m->upd_runs[g];
            if (!runs.empty() && runs.back().second == b) runs.back().second = e;
            else runs.push_back({b, e});
        }
    }

    const size_t nb = (size_t)m->n_arena * sizeof(float);
    ALLOC(m, m->params, nb);
    ALLOC(m, m->grads, nb);
    ALLOC(m, m->adam_m, nb);
    ALLOC(m, m->adam_v, nb);
    if (m->use_bf16) ALLOC(m, m->pbf, (size_t)m->decay_end * sizeof(bf16));
    ALLOC(m, m->st, sizeof(DevState));

    const size_t M = m->M, C = m->C, A = m->act_bytes;
    m->la.resize(m->L);
    for (int l = 0; l < m->L; l++) {
        LayerActs& a = m->la[l];
        ALLOC(m, a.x_in, M * C * 4);
        ALLOC(m, a.x_mid, M * C * 4);
        ALLOC(m, a.u1, M * C * A);
        ALLOC(m, a.mu1, M * 4);
        ALLOC(m, a.rs1, M * 4);
        ALLOC(m, a.qkv, M * 3 * C * A);
        ALLOC(m, a.att, M * C * A);
        ALLOC(m, a.lse, M * m->H * 4);
        ALLOC(m, a.u2, M * C * A);
        ALLOC(m, a.mu2, M * 4);
        ALLOC(m, a.rs2, M * 4);
        ALLOC(m, a.hpre, M * 4 * C * A);
        ALLOC(m, a.hgel, M * 4 * C * A);
    }
    ALLOC(m, m->x_final, M * C * 4);
    ALLOC(m, m->uf, M * C * A);
    ALLOC(m, m->muf, M * 4);
    ALLOC(m, m->rsf, M * 4);
    ALLOC(m, m->logits, M * (size_t)m->Vp * A);
    ALLOC(m, m->row_loss, M * 4);
    ALLOC(m, m->last_logits, (size_t)m->B * m->Vp * 4);

    ALLOC(m, m->dres, M * C * 4);
    if (m->use_bf16) ALLOC(m, m->dres_act, M * C * A);
    else m->dres_act = m->dres;
    ALLOC(m, m->du, M * C * A);
    ALLOC(m, m->dqkv, M * 3 * C * A);
    ALLOC(m, m->datt, M * C * A);
    ALLOC(m, m->yproj, M * C * A);
    ALLOC(m, m->dh, M * 4 * C * A);
    ALLOC(m, m->Dbuf, M * m->H * 4);
    // two buffers: the side stream reduces one while the next row pass fills the other
    ALLOC(m, m->ln_partial, 2 * k::layernorm_bwd_partial_floats(m->M, m->C) * 4);
    size_t cs = k::colsum_partial_floats(m->M, 4 * m->C);
    ALLOC(m, m->cs_partial, cs * 4);
    if (m->use_bf16) ALLOC(m, m->fc_cs_part, (size_t)((m->M + 31) / 32) * 4 * m->C * 4);
    ALLOC(m, m->emb_ws, k::embed_bwd_workspace(m->M, m->C));
    m->norm_parts = 2 * k::num_sms();
    ALLOC(m, m->norm_partial, (size_t)m->norm_parts * sizeof(double));
    // split-K workspace for the weight gradients (tensor-core path)
    if (m->use_bf16) {
        size_t need = 0;
        const int dims[4][2] = {{3 * m->C, m->C}, {m->C, m->C}, {4 * m->C, m->C}, {m->C, 4 * m->C}};
        for (auto& d : dims) {
            int tiles = ((d[0] + 127) / 128) * ((d[1] + (d[1] % 256 == 0 ? 255 : 127)) /
                                                (d[1] % 256 == 0 ? 256 : 128));
            int splits = k::num_sms() / tiles;
            if (splits > 16) splits = 16;
            if (splits > 1) need = std::max(need, (size_t)splits * d[0] * d[1]);
        }
        m->splitk_ws_floats = need;
        if (need) ALLOC(m, m->splitk_ws, need * 4);
    }

    // host init in canonical order, then upload
    std::vector<float> host((size_t)m->n_arena, 0.0f);
    for (size_t k = 0; k < m->tensors.size(); k++)
        host_init_tensor(cfg, m->tensors[k], (int)k, seed, host.data() + m->tensors[k].offset);
    CK(m, cudaMemcpy(m->params, host.data(), nb, cudaMemcpyHostToDevice));
    CK(m, cudaMemset(m->grads, 0, nb));
    CK(m, cudaMemset(m->adam_m, 0, nb));
    CK(m, cudaMemset(m->adam_v, 0, nb));
    CK(m, cudaMemset(m->st, 0, sizeof(DevState)));
    if (m->use_bf16) CK(m, k::f32_to_bf16(m->params, m->pbf, m->decay_end, nullptr));
    CK(m, cudaStreamCreateWithFlags(&m->side, cudaStreamNonBlocking));
    CK(m, cudaDeviceSynchronize());
    return GPT2_OK;
}

// ------------------------------------------------------------------ profiling
// Optional per-site timing: CUDA events recorded on the model's stream around
// each launch site, with the site's algorithmic FLOPs and HBM bytes.
struct ProfRec {
    int site;
    int ev;
    int kernels;
    double flops, bytes;
};

static int site_id(gpt2_model* m, const char* name);
static int prof_begin(gpt2_model* m);
static void prof_end(gpt2_model* m, int ev, const char* site, int kernels, double flops,
                     double bytes);

#define RUN(m, site, nk, flops, bytes, expr)            \
    do {                                                \
        int ev__ = prof_begin(m);                       \
        CK(m, expr);                                    \
        prof_end(m, ev__, site, nk, flops, bytes);      \
    } while (0)

static int site_id(gpt2_model* m, const char* name) {
    for (size_t i = 0; i < m->sites.size(); i++)
        if (m->sites[i].name == name || std::strcmp(m->sites[i].name, name) == 0) return (int)i;
    m->sites.push_back({name, 0, 0, 0.0, 0.0, 0.0});
    return (int)m->sites.size() - 1;
}

static int prof_begin(gpt2_model* m) {
    if (!m->prof_on) return -1;
    while ((int)m->prof_ev.size() < m->prof_next + 2) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return -1;
        m->prof_ev.push_back(e);
    }
    int ev = m->prof_next;
    m->prof_next += 2;
    cudaEventRecord(m->prof_ev[ev], m->stream);
    return ev;
}

static void prof_end(gpt2_model* m, int ev, const char* site, int kernels, double flops,
                     double bytes) {
    int id = site_id(m, site);
    auto& a = m->sites[id];
    a.calls += 1;
    a.kernels += kernels;
    a.flops += flops;
    a.bytes += bytes;
    if (ev >= 0) {
        cudaEventRecord(m->prof_ev[ev + 1], m->stream);
        m->prof_pending.push_back({id, ev});
    }
}

static int prof_collect(gpt2_model* m) {
    CK(m, cudaStreamSynchronize(m->stream));
    for (auto& pr : m->prof_pending) {
        float ms = 0.f;
        CK(m, cudaEventElapsedTime(&ms, m->prof_ev[pr.second], m->prof_ev[pr.second + 1]));
        m->sites[pr.first].ms += ms;
    }
    m->prof_pending.clear();
    m->prof_next = 0;
    return GPT2_OK;
}

// ------------------------------------------------------------------ GEMM dispatch
struct Op {
    gpt2_model* m;
    // D[M,N] = A B^T with epilogue e; `site` names the Linear for profiling.
    int gemm(const char* site, int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& e) {
        const double ab = m->act_bytes;
        double bytes = ab * ((double)M * K + (double)N * K);
        double ob = (e.kind == EPI_RESID || e.kind == EPI_ACCUM_F32) ? 8.0 : (e.kind == EPI_GELU ? 2 * ab : ab);
        if (e.kind == EPI_GELU_BWD) ob = 2 * ab;
        bytes += ob * (double)M * N;
        if (m->use_bf16 && k::gemm_rows_supported(M, N, K, A, B, e))
            // a handful of rows (generation): weight streaming, no tensor-core tiles
            RUN(m, site, 1, 2.0 * M * N * K, bytes, k::gemm_rows_bf16(M, N, K, A, B, e, m->stream));
        else if (m->use_bf16)
            RUN(m, site, 1, 2.0 * M * N * K, bytes, k::gemm_bf16_tc(M, N, K, A, B, e, 1, m->st, m->stream));
        else
            RUN(m, site, 1, 2.0 * M * N * K, bytes, k::gemm_f32(M, N, K, A, B, e, m->stream));
        return GPT2_OK;
    }
    // dW[N_out, K_in] += dY^T X, dY [M, N_out] (ld ldy), X [M, K_in] (ld ldx).
    int gemm_dw(const char* site, int n_out, int k_in, const void* dy, int64_t ldy, const void* x,
                int64_t ldx, float* dW, cudaStream_t s) {
        GemmOperand A{dy, ldy, false}, B{x, ldx, false};
        const int M = m->M;
        const double flops = 2.0 * n_out * k_in * (double)M;
        const double bytes = m->act_bytes * (double)M * (n_out + k_in) + 8.0 * n_out * k_in;
        if (!m->use_bf16) {
            GemmEpi e{EPI_ACCUM_F32, nullptr, dW, k_in, nullptr, 0, nullptr, 0};
            RUN(m, site, 1, flops, bytes, k::gemm_f32(n_out, k_in, M, A, B, e, s));
            return GPT2_OK;
        }
        const int bn = (k_in % 256 == 0 || k_in > 2048) ? 256 : 128;
        // one wave: as many K splits as fit the SMs beside the tiles (floor)
        int tiles = ((n_out + 127) / 128) * ((k_in + bn - 1) / bn);
        int splits = k::num_sms() / tiles;
        if (splits > 16) splits = 16;
        if (splits > 1 && (size_t)splits * n_out * k_in <= m->splitk_ws_floats) {
            GemmEpi e{EPI_STORE_F32, nullptr, m->splitk_ws, k_in, nullptr, 0, nullptr, 0};
            // the launcher lowers `splits` so that every split owns k-blocks
            int kblocks = (M + 63) / 64;
            int kpb = (kblocks + splits - 1) / splits;
            int eff = (kblocks + kpb - 1) / kpb;
            RUN(m, site, 1, flops, bytes - 8.0 * n_out * k_in + 4.0 * eff * n_out * k_in,
                k::gemm_bf16_tc(n_out, k_in, M, A, B, e, splits, m->st, s));
            RUN(m, "splitk_reduce", 1, 0.0, 4.0 * (eff + 2) * n_out * (double)k_in,
                k::splitk_reduce_add(m->splitk_ws, eff, (int64_t)n_out * k_in, dW, s));
            return GPT2_OK;
        }
        GemmEpi e{EPI_ACCUM_F32, nullptr, dW, k_in, nullptr, 0, nullptr, 0};
        RUN(m, site, 1, flops, bytes, k::gemm_bf16_tc(n_out, k_in, M, A, B, e, 1, m->st, s));
        return GPT2_OK;
    }
};

// Cross-stream ordering: mark() records an event on `s` (the work enqueued
// there so far); after(s, e) makes later work on `s` wait for it. Events come
// from a pool that each backward pass reuses from the start: a wait binds to
// the record that precedes it, so re-recording later does not disturb it.
static int xmark(gpt2_model* m, cudaStream_t s, cudaEvent_t* out) {
    if (m->xev_next == (int)m->xev.size()) {
        cudaEvent_t e;
        CK(m, cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        m->xev.push_back(e);
    }
    *out = m->xev[m->xev_next++];
    CK(m, cudaEventRecord(*out, s));
    return GPT2_OK;
}
static int xafter(gpt2_model* m, cudaStream_t s, cudaEvent_t e) {
    if (e) CK(m, cudaStreamWaitEvent(s, e, 0));
    return GPT2_OK;
}
// The model's stream waits for everything enqueued on the side stream.
static int join_side(gpt2_model* m) {
    if (!m->upd_pending) return GPT2_OK;
    m->upd_pending = false;
    cudaEvent_t e;
    int r = xmark(m, m->side, &e);
    if (r) return r;
    return xafter(m, m->stream, e);
}
// Before the forward reads parameter group g: wait for its AdamW update.
static int param_wait(gpt2_model* m, int g) {
    return m->upd_pending ? xafter(m, m->stream, m->upd_ev[g]) : GPT2_OK;
}

#define OPR(expr)                 \
    do {                          \
        int r__ = (expr);         \
        if (r__) return r__;      \
    } while (0)

// causal attention algorithmic FLOPs: two T x T x hs products over the
// visible (i, j <= i) pairs forward; five in the backward (S recomputed, dV,
// dP, dQ, dK).
static double attn_flops(const gpt2_model* m, int products) {
    double pairs = (double)m->T * (m->T + 1) / 2.0;
    return 2.0 * products * pairs * m->hs * (double)m->B * m->H;
}

// last_t > 0: generation's forward, the LM head only on position last_t - 1 of
// every sequence, into m->last_logits (no loss).
template <typename Act>
static int forward_impl(gpt2_model* m, const int32_t* tok, const int32_t* tgt, int last_t = 0) {
    cudaStream_t s = m->stream;
    const int M = m->M, C = m->C, L = m->L, T = m->T, B = m->B, H = m->H;
    const double A = m->act_bytes, MC = (double)M * C;
    Op op{m};
    RUN(m, "validate", 1, 0, 8.0 * M, k::validate_inputs(tok, tgt, M, m->V, m->st, m->accum, s));
    OPR(param_wait(m, 0));
    RUN(m, "embed_fwd", 1, 0, 4.0 * M + 12.0 * MC,
        k::embed_fwd(tok, m->P(0), m->P(1), m->la[0].x_in, M, T, C, m->V, s));
    // LayerNorm: read x, write u, mu, rstd; fused residual add: also read y, write x
    const double ln_bytes = MC * (4 + A) + 8.0 * M;
    const double add_ln_bytes = ln_bytes + MC * (A + 4);
    OPR(param_wait(m, 1));
    RUN(m, "layernorm_fwd", 1, 0, ln_bytes,
        k::layernorm_fwd<Act>(m->la[0].x_in, nullptr, nullptr, m->P(m->lt(0, T_LN1G)),
                              m->P(m->lt(0, T_LN1B)), (Act*)m->la[0].u1, m->la[0].mu1, m->la[0].rs1,
                              M, C, s));
    for (int l = 0; l < L; l++) {
        LayerActs& a = m->la[l];
        {
            GemmEpi e{EPI_STORE_ACT, m->P(m->lt(l, T_ATTB)), a.qkv, 3 * C, nullptr, 0, nullptr, 0};
            OPR(op.gemm("gemm_qkv_fwd", M, 3 * C, C, {a.u1, C, true}, {m->W(m->lt(l, T_ATTW)), C, true}, e));
        }
        if (m->use_bf16)
            RUN(m, "attention_fwd", 1, attn_flops(m, 2), MC * A * 4,
                k::attention_fwd_bf16((const bf16*)a.qkv, (bf16*)a.att, a.lse, B, T, H, m->hs, m->st, s));
        else
            RUN(m, "attention_fwd", 1, attn_flops(m, 2), MC * A * 4,
                k::attention_fwd_f32((const float*)a.qkv, (float*)a.att, a.lse, B, T, H, m->hs, s));
        {
            // y = att W_ap^T + b_ap; x_mid = x_in + y fused into ln_2
            GemmEpi e{EPI_STORE_ACT, m->P(m->lt(l, T_APB)), m->yproj, C, nullptr, 0, nullptr, 0};
            OPR(op.gemm("gemm_attproj_fwd", M, C, C, {a.att, C, true}, {m->W(m->lt(l, T_APW)), C, true}, e));
        }
        RUN(m, "layernorm_fwd", 1, 0, add_ln_bytes,
            k::layernorm_fwd<Act>(a.x_in, (const Act*)m->yproj, a.x_mid, m->P(m->lt(l, T_LN2G)),
                                  m->P(m->lt(l, T_LN2B)), (Act*)a.u2, a.mu2, a.rs2, M, C, s));
        {
            GemmEpi e{EPI_GELU, m->P(m->lt(l, T_FCB)), a.hpre, 4 * C, a.hgel, 4 * C, nullptr, 0};
            OPR(op.gemm("gemm_fc_fwd", M, 4 * C, C, {a.u2, C, true}, {m->W(m->lt(l, T_FCW)), C, true}, e));
        }
        {
            // y = gelu(h) W_mp^T + b_mp; the next residual x_mid + y is fused into
            // the next block's ln_1 (or ln_f)
            GemmEpi e{EPI_STORE_ACT, m->P(m->lt(l, T_MPB)), m->yproj, C, nullptr, 0, nullptr, 0};
            OPR(op.gemm("gemm_mlpproj_fwd", M, C, 4 * C, {a.hgel, 4 * C, true},
                        {m->W(m->lt(l, T_MPW)), 4 * C, true}, e));
        }
        if (l + 1 < L) {
            LayerActs& n = m->la[l + 1];
            OPR(param_wait(m, l + 2));
            RUN(m, "layernorm_fwd", 1, 0, add_ln_bytes,
                k::layernorm_fwd<Act>(a.x_mid, (const Act*)m->yproj, n.x_in, m->P(m->lt(l + 1, T_LN1G)),
                                      m->P(m->lt(l + 1, T_LN1B)), (Act*)n.u1, n.mu1, n.rs1, M, C, s));
        }
    }
    OPR(param_wait(m, L + 1));
    m->upd_pending = false;      // every group has been waited for
    RUN(m, "layernorm_fwd", 1, 0, add_ln_bytes,
        k::layernorm_fwd<Act>(m->la[L - 1].x_mid, (const Act*)m->yproj, m->x_final, m->P(m->lnf_g()),
                              m->P(m->lnf_g() + 1), (Act*)m->uf, m->muf, m->rsf, M, C, s));
    m->kv_len = last_t;           // training forwards (last_t == 0) overwrite the cache
    if (last_t > 0) {
        // the tied head on one position per sequence: rows b*T + last_t - 1 of uf
        const void* a = (const char*)m->uf + (size_t)(last_t - 1) * C * m->act_bytes;
        GemmEpi e{EPI_STORE_F32, nullptr, m->last_logits, m->Vp, nullptr, 0, nullptr, 0};
        OPR(op.gemm("gemm_lmhead_last", B, m->Vp, C, {a, (int64_t)T * C, true}, {m->W(0), C, true}, e));
        return GPT2_OK;
    }
    {
        // tied LM head: logits = uf wte^T over all Vp rows of wte (pad columns
        // are masked by the cross-entropy)
        GemmEpi e{EPI_STORE_ACT, nullptr, m->logits, m->Vp, nullptr, 0, nullptr, 0};
        OPR(op.gemm("gemm_lmhead_fwd", M, m->Vp, C, {m->uf, C, true}, {m->W(0), C, true}, e));
    }
    if (tgt) {
        RUN(m, "cross_entropy", 1, 0, 2.0 * A * M * m->Vp + 8.0 * M,
            k::cross_entropy<Act>((Act*)m->logits, tgt, m->row_loss, M, m->V, m->Vp, m->st, s));
        RUN(m, "loss_reduce", 1, 0, 4.0 * M, k::loss_reduce(m->row_loss, M, m->st, s));
    }
    return GPT2_OK;
}

// One decoding step: the forward of position p = t - 1 of every sequence
// alone, its query attending to the cached keys and values of positions
// 0..p (this step writes row p of every layer's qkv buffer), the head on the
// new row into m->last_logits. Row buffers (B rows each): residual stream x0,
// x1 (fp32 [B, C]), LayerNorm statistics, u, att, y (act [B, C]), gelu'(pre)
// and gelu(pre) (act [B, 4C]).
template <typename Act>
static int decode_impl(gpt2_model* m, const int32_t* tok, int t) {
    cudaStream_t s = m->stream;
    const int C = m->C, L = m->L, T = m->T, B = m->B, H = m->H, p = t - 1;
    const double A = m->act_bytes, BC = (double)B * C;
    Op op{m};
    auto carve = [](char*& q, size_t bytes) {
        char* r = q;
        q += (bytes + 255) / 256 * 256;
        return (void*)r;
    };
    char* q = (char*)m->dec_ws;
    float* x0 = (float*)carve(q, (size_t)B * C * 4);
    float* x1 = (float*)carve(q, (size_t)B * C * 4);
    float* mu = (float*)carve(q, (size_t)B * 4);
    float* rs = (float*)carve(q, (size_t)B * 4);
    Act* u = (Act*)carve(q, (size_t)B * C * sizeof(Act));
    Act* att = (Act*)carve(q, (size_t)B * C * sizeof(Act));
    Act* y = (Act*)carve(q, (size_t)B * C * sizeof(Act));
    Act* hpre = (Act*)carve(q, (size_t)B * 4 * C * sizeof(Act));
    Act* hgel = (Act*)carve(q, (size_t)B * 4 * C * sizeof(Act));
    float* part = (float*)carve(q, k::attention_decode_workspace_floats(B, T, H, m->hs) * 4);
    const double ln_bytes = BC * (4 + A) + 8.0 * B, add_ln_bytes = ln_bytes + BC * (A + 4);
    RUN(m, "decode_embed", 1, 0, 4.0 * B + 12.0 * BC,
        k::embed_rows(tok, m->P(0), m->P(1), x0, B, p, C, m->V, m->st, s));
    RUN(m, "decode_layernorm", 1, 0, ln_bytes,
        k::layernorm_fwd<Act>(x0, nullptr, nullptr, m->P(m->lt(0, T_LN1G)), m->P(m->lt(0, T_LN1B)), u, mu, rs,
                              B, C, s));
    for (int l = 0; l < L; l++) {
        LayerActs& a = m->la[l];
        {
            // q, k, v of the new row go to row p of the layer's qkv buffer
            Act* qkv_p = (Act*)a.qkv + (size_t)p * 3 * C;
            GemmEpi e{EPI_STORE_ACT, m->P(m->lt(l, T_ATTB)), qkv_p, (int64_t)T * 3 * C, nullptr, 0, nullptr, 0};
            OPR(op.gemm("decode_gemm_qkv", B, 3 * C, C, {u, C, true}, {m->W(m->lt(l, T_ATTW)), C, true}, e));
        }
        RUN(m, "decode_attention", 1, 4.0 * (p + 1) * m->hs * (double)B * H, 2.0 * A * (p + 1) * BC,
            k::attention_decode<Act>((const Act*)a.qkv, att, part, B, T, H, m->hs, p, s));
        {
            GemmEpi e{EPI_STORE_ACT, m->P(m->lt(l, T_APB)), y, C, nullptr, 0, nullptr, 0};
            OPR(op.gemm("decode_gemm_attproj", B, C, C, {att, C, true}, {m->W(m->lt(l, T_APW)), C, true}, e));
        }
        RUN(m, "decode_layernorm", 1, 0, add_ln_bytes,
            k::layernorm_fwd<Act>(x0, y, x1, m->P(m->lt(l, T_LN2G)), m->P(m->lt(l, T_LN2B)), u, mu, rs, B, C, s));
        {
            GemmEpi e{EPI_GELU, m->P(m->lt(l, T_FCB)), hpre, 4 * C, hgel, 4 * C, nullptr, 0};
            OPR(op.gemm("decode_gemm_fc", B, 4 * C, C, {u, C, true}, {m->W(m->lt(l, T_FCW)), C, true}, e));
        }
        {
            GemmEpi e{EPI_STORE_ACT, m->P(m->lt(l, T_MPB)), y, C, nullptr, 0, nullptr, 0};
            OPR(op.gemm("decode_gemm_mlpproj", B, C, 4 * C, {hgel, 4 * C, true},
                        {m->W(m->lt(l, T_MPW)), 4 * C, true}, e));
        }
        // x0 = x1 + y, and the next LayerNorm (ln_1 of block l + 1, or ln_f)
        const bool last = l + 1 == L;
        RUN(m, "decode_layernorm", 1, 0, add_ln_bytes,
            k::layernorm_fwd<Act>(x1, y, x0, m->P(last ? m->lnf_g() : m->lt(l + 1, T_LN1G)),
                                  m->P(last ? m->lnf_g() + 1 : m->lt(l + 1, T_LN1B)), u, mu, rs, B, C, s));
    }
    GemmEpi e{EPI_STORE_F32, nullptr, m->last_logits, m->Vp, nullptr, 0, nullptr, 0};
    OPR(op.gemm("decode_gemm_lmhead", B, m->Vp, C, {u, C, true}, {m->W(0), C, true}, e));
    m->kv_len = t;
    return GPT2_OK;
}

template <typename Act>
static int backward_impl(gpt2_model* m) {
    cudaStream_t s = m->stream;
    const int M = m->M, C = m->C, L = m->L, T = m->T, B = m->B, H = m->H, Vp = m->Vp;
    const double A = m->act_bytes, MC = (double)M * C;
    Op op{m};
    // LN backward: read du, x, read+write dres (first call writes only), write dres_act
    auto ln_bytes = [&](bool acc) { return MC * (A + 4 + (acc ? 8 : 4) + (m->use_bf16 ? A : 0)); };
    // Weight-gradient work goes to the side stream (the main one when
    // profiling, so that every site is timed alone). The main chain waits
    // for the side only where a buffer the side still reads is overwritten:
    // dres_act (read by the dW of the two residual projections), dh (dW and
    // bias of fc), dqkv (dW and bias of the qkv projection).
    const bool fork = m->side && !m->prof_on;
    cudaStream_t s2 = fork ? m->side : s;
    m->xev_next = 0;
    cudaEvent_t ev = nullptr, dh_free = nullptr, dqkv_free = nullptr, dres_free = nullptr;
    auto to_side = [&]() -> int {            // side waits for everything on main so far
        if (!fork) return GPT2_OK;
        OPR(xmark(m, s, &ev));
        return xafter(m, s2, ev);
    };
    auto side_done = [&](cudaEvent_t* e) -> int {
        if (!fork) return GPT2_OK;
        return xmark(m, s2, e);
    };
    auto main_after = [&](cudaEvent_t e) -> int { return fork ? xafter(m, s, e) : GPT2_OK; };
    // LayerNorm backward: the row pass on the main chain; the reduction of its
    // per-block partials into dgamma, dbeta and the preceding projection's bias
    // gradient on the side, from one of two alternating partials buffers
    const size_t ln_pf = k::layernorm_bwd_partial_floats(M, C);
    cudaEvent_t ln_free[2] = {nullptr, nullptr};
    int ln_iter = 0;
    auto ln_bwd = [&](const float* x, int gi, const float* mu, const float* rs, bool acc,
                      float* dsum) -> int {
        float* part = m->ln_partial + (size_t)(ln_iter & 1) * ln_pf;
        OPR(main_after(ln_free[ln_iter & 1]));
        RUN(m, "layernorm_bwd", 1, 0, ln_bytes(acc),
            k::layernorm_bwd_rows<Act>((const Act*)m->du, x, m->P(gi), mu, rs, m->dres, (Act*)m->dres_act,
                                       acc, dsum != nullptr, M, C, part, s));
        OPR(to_side());
        RUN(m, "ln_param_reduce", 1, 0, 4.0 * ln_pf + 12.0 * C,
            k::layernorm_bwd_params(part, M, C, m->G(gi), m->G(gi + 1), dsum, s2));
        OPR(side_done(&ln_free[ln_iter & 1]));
        ln_iter++;
        return GPT2_OK;
    };
    // LM head: du = dz wte ; dwte += dz^T uf. The side also sorts the token ids
    // for the embedding backward (they depend on nothing else).
    {
        GemmEpi e{EPI_STORE_ACT, nullptr, m->du, C, nullptr, 0, nullptr, 0};
        OPR(to_side());
        RUN(m, "embed_bwd", 1, 0, 8.0 * M, k::embed_bwd_sort(m->last_tok, M, m->V, m->emb_ws, s2));
        OPR(op.gemm_dw("gemm_lmhead_dw", Vp, C, m->logits, Vp, m->uf, C, m->G(0), s2));
        OPR(op.gemm("gemm_lmhead_dx", M, C, Vp, {m->logits, Vp, true}, {m->W(0), C, false}, e));
    }
    // the new dres is the output gradient of the last MLP projection: its
    // column sums (that projection's bias gradient) come out of the same pass
    OPR(ln_bwd(m->x_final, m->lnf_g(), m->muf, m->rsf, false, m->G(m->lt(L - 1, T_MPB))));
    for (int l = L - 1; l >= 0; l--) {
        LayerActs& a = m->la[l];
        // MLP projection: x_out = x_mid + hgel W_mp^T + b_mp
        {
            // bf16: the GEMM also leaves the column sums of dh (fc's bias
            // gradient) per 32-row group in fc_cs_part
            GemmEpi e{EPI_GELU_BWD, nullptr, m->dh, 4 * C, m->use_bf16 ? m->fc_cs_part : nullptr, 4 * C,
                      a.hpre, 4 * C};
            OPR(to_side());
            OPR(op.gemm_dw("gemm_mlpproj_dw", C, 4 * C, m->dres_act, C, a.hgel, 4 * C,
                           m->G(m->lt(l, T_MPW)), s2));
            OPR(side_done(&dres_free));
            OPR(main_after(dh_free));
            OPR(op.gemm("gemm_mlpproj_dx", M, 4 * C, C, {m->dres_act, C, true},
                        {m->W(m->lt(l, T_MPW)), 4 * C, false}, e));
        }
        // fc: hpre = u2 W_fc^T + b_fc
        {
            GemmEpi e{EPI_STORE_ACT, nullptr, m->du, C, nullptr, 0, nullptr, 0};
            OPR(to_side());
            OPR(op.gemm_dw("gemm_fc_dw", 4 * C, C, m->dh, 4 * C, a.u2, C, m->G(m->lt(l, T_FCW)), s2));
            if (m->use_bf16) {
                const int groups = (M + 31) / 32;
                RUN(m, "bias_colsum", 1, 0, 4.0 * groups * 4 * C,
                    k::colsum_partials_add(m->fc_cs_part, groups, 4 * C, m->G(m->lt(l, T_FCB)), s2));
            } else {
                RUN(m, "bias_colsum", 2, 0, 4.0 * MC * A,
                    k::colsum_add<Act>((const Act*)m->dh, 4 * C, M, 4 * C, m->G(m->lt(l, T_FCB)),
                                       m->cs_partial, s2));
            }
            OPR(side_done(&dh_free));
            OPR(op.gemm("gemm_fc_dx", M, C, 4 * C, {m->dh, 4 * C, true}, {m->W(m->lt(l, T_FCW)), C, false}, e));
        }
        OPR(main_after(dres_free));
        OPR(ln_bwd(a.x_mid, m->lt(l, T_LN2G), a.mu2, a.rs2, true, m->G(m->lt(l, T_APB))));
        // attention projection: x_mid = x_in + att W_ap^T + b_ap
        {
            GemmEpi e{EPI_STORE_ACT, nullptr, m->datt, C, nullptr, 0, nullptr, 0};
            OPR(to_side());
            OPR(op.gemm_dw("gemm_attproj_dw", C, C, m->dres_act, C, a.att, C, m->G(m->lt(l, T_APW)), s2));
            OPR(side_done(&dres_free));
            OPR(op.gemm("gemm_attproj_dx", M, C, C, {m->dres_act, C, true}, {m->W(m->lt(l, T_APW)), C, false}, e));
        }
        OPR(main_after(dqkv_free));
        if (m->use_bf16)
            RUN(m, "attention_bwd", 2, attn_flops(m, 5), MC * A * 8,
                k::attention_bwd_bf16((const bf16*)a.qkv, (const bf16*)a.att, a.lse, (const bf16*)m->datt,
                                      (bf16*)m->dqkv, m->Dbuf, B, T, H, m->hs, m->st, s));
        else
            RUN(m, "attention_bwd", 3, attn_flops(m, 5), MC * A * 8,
                k::attention_bwd_f32((const float*)a.qkv, (const float*)a.att, a.lse, (const float*)m->datt,
                                     (float*)m->dqkv, m->Dbuf, B, T, H, m->hs, s));
        // qkv: qkv = u1 W_attn^T + b_attn
        {
            GemmEpi e{EPI_STORE_ACT, nullptr, m->du, C, nullptr, 0, nullptr, 0};
            OPR(to_side());
            OPR(op.gemm_dw("gemm_qkv_dw", 3 * C, C, m->dqkv, 3 * C, a.u1, C, m->G(m->lt(l, T_ATTW)), s2));
            RUN(m, "bias_colsum", 2, 0, 3.0 * MC * A,
                k::colsum_add<Act>((const Act*)m->dqkv, 3 * C, M, 3 * C, m->G(m->lt(l, T_ATTB)),
                                   m->cs_partial, s2));
            OPR(side_done(&dqkv_free));
            OPR(op.gemm("gemm_qkv_dx", M, C, 3 * C, {m->dqkv, 3 * C, true}, {m->W(m->lt(l, T_ATTW)), C, false}, e));
        }
        OPR(main_after(dres_free));
        OPR(ln_bwd(a.x_in, m->lt(l, T_LN1G), a.mu1, a.rs1, true,
                   l > 0 ? m->G(m->lt(l - 1, T_MPB)) : nullptr));
    }
    // join: the tied embedding's gradient also receives the LM head's dW
    if (fork) {
        OPR(xmark(m, s2, &ev));
        OPR(xafter(m, s, ev));
    }
    RUN(m, "embed_bwd", 3, 0, 8.0 * MC,
        k::embed_bwd_apply(m->dres, m->G(0), m->G(1), M, T, C, m->emb_ws, s));
    return GPT2_OK;
}

static int check_device_status(gpt2_model* m) {
    DevState st;
    CK(m, cudaMemcpyAsync(&st, m->st, sizeof(DevState), cudaMemcpyDeviceToHost, m->stream));
    CK(m, cudaStreamSynchronize(m->stream));
    if (st.err) {
        unsigned zero = 0;
        CK(m, cudaMemcpy(&m->st->err, &zero, sizeof(unsigned), cudaMemcpyHostToDevice));
        if (st.err & ERR_TIMEOUT)
            return fail(m, GPT2_ETIMEOUT, "a bounded device wait expired (site " +
                                              std::to_string(st.timeout_site) + ")");
        if (st.err & ERR_TOKEN_RANGE) return fail(m, GPT2_ERANGE, "token id outside [0, vocab_size)");
        return fail(m, GPT2_ERANGE, "target id outside [0, vocab_size) and not -1");
    }
    return GPT2_OK;
}

// ------------------------------------------------------------------ C ABI
extern "C" {

const char* gpt2_version(void) { return GPT2_VERSION; }

const char* gpt2_last_error(const gpt2_model* m) {
    return m ? m->err.c_str() : g_create_error.c_str();
}

int gpt2_create(const gpt2_config* cfg, uint64_t seed, gpt2_model** out) {
    if (!out) return fail(nullptr, GPT2_EINVAL, "out is NULL");
    *out = nullptr;
    std::string why;
    int r = validate_cfg(cfg, why);
    if (r) return fail(nullptr, r, why);
    gpt2_model* m = new gpt2_model();
    r = create_impl(m, cfg, seed);
    if (r) {
        g_create_error = m->err;
        gpt2_destroy(m);
        return r;
    }
    *out = m;
    return GPT2_OK;
}

void gpt2_destroy(gpt2_model* m) {
    if (!m) return;
    cudaDeviceSynchronize();
    for (cudaEvent_t e : m->prof_ev) cudaEventDestroy(e);
    for (cudaEvent_t e : m->xev) cudaEventDestroy(e);
    for (cudaEvent_t e : m->upd_ev) cudaEventDestroy(e);
    if (m->side) cudaStreamDestroy(m->side);
    for (void* p : m->allocs) cudaFree(p);
    delete m;
}

int gpt2_set_stream(gpt2_model* m, void* stream) {
    if (!m) return GPT2_EINVAL;
    int r = join_side(m);
    if (r) return r;
    m->stream = (cudaStream_t)stream;
    return GPT2_OK;
}

int gpt2_forward(gpt2_model* m, const int32_t* tok, const int32_t* tgt, float* h_loss) {
    if (!m) return GPT2_EINVAL;
    if (!tok) return fail(m, GPT2_EINVAL, "tokens pointer is NULL");
    int r = m->use_bf16 ? forward_impl<bf16>(m, tok, tgt) : forward_impl<float>(m, tok, tgt);
    m->have_targets = false;
    if (r) return r;
    m->last_tok = tok;
    m->have_targets = tgt != nullptr;
    if (h_loss) {
        if (!tgt) return fail(m, GPT2_EINVAL, "h_loss requested without targets");
        return gpt2_get_loss(m, h_loss);
    }
    return GPT2_OK;
}

int gpt2_forward_last(gpt2_model* m, const int32_t* tok, int t, float* d_logits) {
    if (!m) return GPT2_EINVAL;
    if (!tok || !d_logits) return fail(m, GPT2_EINVAL, "tokens or logits pointer is NULL");
    if (t < 1 || t > m->T) return fail(m, GPT2_EINVAL, "t must be in [1, seq_len]");
    m->have_targets = false;
    int r = m->use_bf16 ? forward_impl<bf16>(m, tok, nullptr, t) : forward_impl<float>(m, tok, nullptr, t);
    if (r) return r;
    m->last_tok = tok;
    CK(m, cudaMemcpy2DAsync(d_logits, (size_t)m->V * 4, m->last_logits, (size_t)m->Vp * 4, (size_t)m->V * 4,
                            (size_t)m->B, cudaMemcpyDeviceToDevice, m->stream));
    return GPT2_OK;
}

int gpt2_decode_step(gpt2_model* m, const int32_t* tok, int t, float* d_logits) {
    if (!m) return GPT2_EINVAL;
    if (!tok || !d_logits) return fail(m, GPT2_EINVAL, "tokens or logits pointer is NULL");
    if (t < 1 || t > m->T) return fail(m, GPT2_EINVAL, "t must be in [1, seq_len]");
    if (m->hs > 128) return fail(m, GPT2_EINVAL, "decoding needs a head size of at most 128");
    if (t - 1 > m->kv_len)
        return fail(m, GPT2_ESTATE, "the key/value cache does not hold positions 0..t-2: run gpt2_forward_last first");
    if (int r = join_side(m)) return r;
    if (!m->dec_ws) {
        const size_t rows = (size_t)m->B, C = (size_t)m->C;
        const size_t bytes = 2 * (rows * C * 4 + 256) + 2 * (rows * 4 + 256) + 3 * (rows * C * m->act_bytes + 256) +
                             2 * (rows * 4 * C * m->act_bytes + 256) +
                             k::attention_decode_workspace_floats(m->B, m->T, m->H, m->hs) * 4 + 256;
        ALLOC(m, m->dec_ws, bytes);
    }
    m->have_targets = false;
    int r = m->use_bf16 ? decode_impl<bf16>(m, tok, t) : decode_impl<float>(m, tok, t);
    if (r) return r;
    CK(m, cudaMemcpy2DAsync(d_logits, (size_t)m->V * 4, m->last_logits, (size_t)m->Vp * 4, (size_t)m->V * 4,
                            (size_t)m->B, cudaMemcpyDeviceToDevice, m->stream));
    return GPT2_OK;
}

int gpt2_backward(gpt2_model* m) {
    if (!m) return GPT2_EINVAL;
    {
        int r = join_side(m);
        if (r) return r;
    }
    if (!m->have_targets) return fail(m, GPT2_ESTATE, "backward needs a forward with targets");
    m->have_targets = false;   // the logits buffer now holds consumed gradients
    return m->use_bf16 ? backward_impl<bf16>(m) : backward_impl<float>(m);
}

int gpt2_step(gpt2_model* m, float lr, float beta1, float beta2, float eps, float weight_decay,
              float clip, float* h_grad_norm) {
    if (!m) return GPT2_EINVAL;
    {
        int r = join_side(m);
        if (r) return r;
    }
    cudaStream_t s = m->stream;
    const double n = (double)m->n_arena;
    m->kv_len = 0;                // the parameters change
    RUN(m, "grad_norm", 1, 0, 4.0 * n,
        k::grad_norm(m->grads, m->n_arena, m->norm_partial, m->norm_parts, s));
    RUN(m, "step_finalize", 1, 0, 8.0 * m->norm_parts,
        k::step_finalize(m->norm_partial, m->norm_parts, clip, beta1, beta2, m->st, s));
    bf16* pbf = m->use_bf16 ? m->pbf : nullptr;
    if (!m->side || m->prof_on) {
        RUN(m, "adamw", 1, 0, 28.0 * n + (m->use_bf16 ? 2.0 * m->decay_end : 0.0),
            k::adamw(m->params, m->grads, m->adam_m, m->adam_v, pbf, m->n_arena, m->decay_end,
                     m->decay_end, lr, beta1, beta2, eps, weight_decay, m->st, s));
    } else {
        // on the side stream, group by group (update_groups: contiguous arena
        // runs of the embeddings, each layer, the final LayerNorm)
        cudaEvent_t e;
        int r = xmark(m, s, &e);
        if (r) return r;
        r = xafter(m, m->side, e);
        if (r) return r;
        const int G = m->L + 2;
        while ((int)m->upd_ev.size() < G) {
            cudaEvent_t u;
            CK(m, cudaEventCreateWithFlags(&u, cudaEventDisableTiming));
            m->upd_ev.push_back(u);
        }
        for (int g = 0; g < G; g++) {
            for (const auto& run : m->upd_runs[g]) {
                const int64_t a = run.first, cnt = run.second - run.first;
                const int64_t dend = std::max<int64_t>(0, std::min<int64_t>(cnt, m->decay_end - a));
                RUN(m, "adamw", 1, 0, 28.0 * cnt + (m->use_bf16 ? 2.0 * dend : 0.0),
                    k::adamw(m->params + a, m->grads + a, m->adam_m + a, m->adam_v + a,
                             pbf ? pbf + a : nullptr, cnt, dend, dend, lr, beta1, beta2, eps,
                             weight_decay, m->st, m->side));
            }
            CK(m, cudaEventRecord(m->upd_ev[g], m->side));
        }
        m->upd_pending = true;
    }
    if (h_grad_norm) {
        int r = check_device_status(m);
        if (r) return r;
        DevState st;
        CK(m, cudaMemcpy(&st, m->st, sizeof(DevState), cudaMemcpyDeviceToHost));
        *h_grad_norm = st.grad_norm;
        if (st.skip) return fail(m, GPT2_ENONFINITE, "non-finite gradient norm: update skipped");
    }
    return GPT2_OK;
}

int gpt2_zero_grad(gpt2_model* m) {
    if (!m) return GPT2_EINVAL;
    // behind a pending AdamW (which reads the gradients) on the side stream;
    // the backward writes gradients only on the side stream, or on the model's
    // stream after joining it
    RUN(m, "zero_grad", 0, 0, 4.0 * m->n_arena,
        cudaMemsetAsync(m->grads, 0, (size_t)m->n_arena * sizeof(float),
                        m->upd_pending ? m->side : m->stream));
    return GPT2_OK;
}

double gpt2_lr_schedule(int64_t it, int64_t warmup, int64_t horizon, double lr_max, double lr_min) {
    if (it < warmup) return lr_max * (double)(it + 1) / (double)warmup;
    if (it > horizon) return lr_min;
    double ratio = (double)(it - warmup) / (double)(horizon - warmup);
    return lr_min + 0.5 * (1.0 + std::cos(PI_D * ratio)) * (lr_max - lr_min);
}

int gpt2_sync(gpt2_model* m) {
    if (!m) return GPT2_EINVAL;
    int r = join_side(m);
    if (r) return r;
    return check_device_status(m);
}

int gpt2_join(gpt2_model* m) {
    if (!m) return GPT2_EINVAL;
    return join_side(m);
}

int gpt2_set_wait_limit(gpt2_model* m, unsigned int cycles) {
    if (!m) return GPT2_EINVAL;
    if (int r0 = join_side(m)) return r0;
    CK(m, cudaStreamSynchronize(m->stream));
    CK(m, cudaMemcpy((char*)m->st + offsetof(DevState, wait_limit), &cycles, sizeof cycles,
                     cudaMemcpyHostToDevice));
    return GPT2_OK;
}

int gpt2_get_loss(gpt2_model* m, float* h_loss) {
    if (!m || !h_loss) return GPT2_EINVAL;
    // the loss comes from the forward on the model's stream: no need to wait
    // for a pending parameter update on the side stream
    int r = check_device_status(m);
    if (r) return r;
    DevState st;
    CK(m, cudaMemcpy(&st, m->st, sizeof(DevState), cudaMemcpyDeviceToHost));
    *h_loss = st.loss;
    return GPT2_OK;
}

int gpt2_get_loss_async(gpt2_model* m, float* h_loss) {
    if (!m || !h_loss) return GPT2_EINVAL;
    CK(m, cudaMemcpyAsync(h_loss, &m->st->loss, sizeof(float), cudaMemcpyDeviceToHost, m->stream));
    return GPT2_OK;
}

int gpt2_num_tensors(const gpt2_model* m) { return m ? (int)m->tensors.size() : GPT2_EINVAL; }

int gpt2_tensor_info(const gpt2_model* m, int i, const char** name, int* ndim, int64_t shape[2],
                     int* decays) {
    if (!m || i < 0 || i >= (int)m->tensors.size()) return GPT2_EINVAL;
    const TensorRec& r = m->tensors[i];
    if (name) *name = r.name.c_str();
    if (ndim) *ndim = r.ndim;
    if (shape) { shape[0] = r.shape[0]; shape[1] = r.shape[1]; }
    if (decays) *decays = r.decays ? 1 : 0;
    return GPT2_OK;
}

static float* buffer_of(gpt2_model* m, int which) {
    switch (which) {
        case GPT2_PARAM: return m->params;
        case GPT2_GRAD: return m->grads;
        case GPT2_ADAM_M: return m->adam_m;
        case GPT2_ADAM_V: return m->adam_v;
    }
    return nullptr;
}

int gpt2_copy_tensor(gpt2_model* m, int i, int which, float* dst) {
    if (!m || !dst || i < 0 || i >= (int)m->tensors.size()) return GPT2_EINVAL;
    if (int r0 = join_side(m)) return r0;
    float* buf = buffer_of(m, which);
    if (!buf) return fail(m, GPT2_EINVAL, "unknown buffer selector");
    if (which == GPT2_PARAM) m->kv_len = 0;
    CK(m, cudaStreamSynchronize(m->stream));
    const TensorRec& r = m->tensors[i];
    CK(m, cudaMemcpy(dst, buf + r.offset, r.numel * sizeof(float), cudaMemcpyDeviceToHost));
    return GPT2_OK;
}

int gpt2_set_tensor(gpt2_model* m, int i, int which, const float* src) {
    if (!m || !src || i < 0 || i >= (int)m->tensors.size()) return GPT2_EINVAL;
    if (int r0 = join_side(m)) return r0;
    float* buf = buffer_of(m, which);
    if (!buf) return fail(m, GPT2_EINVAL, "unknown buffer selector");
    CK(m, cudaStreamSynchronize(m->stream));
    const TensorRec& r = m->tensors[i];
    CK(m, cudaMemcpy(buf + r.offset, src, r.numel * sizeof(float), cudaMemcpyHostToDevice));
    if (which == GPT2_PARAM && m->use_bf16 && r.offset < m->decay_end) {
        int64_t n = (r.numel + 63) / 64 * 64;
        CK(m, k::f32_to_bf16(m->params + r.offset, m->pbf + r.offset, n, nullptr));
    }
    CK(m, cudaDeviceSynchronize());
    return GPT2_OK;
}

int gpt2_copy_logits(gpt2_model* m, int64_t row0, int64_t nrows, float* dst) {
    if (!m || !dst || row0 < 0 || nrows < 0 || row0 + nrows > m->M) return GPT2_EINVAL;
    if (int r0 = join_side(m)) return r0;
    CK(m, cudaStreamSynchronize(m->stream));
    const int Vp = m->Vp, V = m->V;
    if (!m->use_bf16) {
        CK(m, cudaMemcpy2D(dst, (size_t)V * 4, (const float*)m->logits + row0 * Vp, (size_t)Vp * 4,
                           (size_t)V * 4, (size_t)nrows, cudaMemcpyDeviceToHost));
        return GPT2_OK;
    }
    std::vector<uint16_t> tmp((size_t)nrows * V);
    CK(m, cudaMemcpy2D(tmp.data(), (size_t)V * 2, (const bf16*)m->logits + row0 * Vp, (size_t)Vp * 2,
                       (size_t)V * 2, (size_t)nrows, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < tmp.size(); i++) {
        uint32_t u = (uint32_t)tmp[i] << 16;
        std::memcpy(&dst[i], &u, 4);
    }
    return GPT2_OK;
}

int gpt2_copy_row_losses(gpt2_model* m, int64_t row0, int64_t nrows, float* dst) {
    if (!m || !dst || row0 < 0 || nrows < 0 || row0 + nrows > m->M) return GPT2_EINVAL;
    if (int r0 = join_side(m)) return r0;
    CK(m, cudaStreamSynchronize(m->stream));
    CK(m, cudaMemcpy(dst, m->row_loss + row0, nrows * sizeof(float), cudaMemcpyDeviceToHost));
    return GPT2_OK;
}

// ------------------------------------------------------------------ checkpoint
static const char CKPT_MAGIC[16] = {'G', 'P', 'T', '2', 'B', '3', '0', '0', 'C', 'K', 'P', 'T', 0, 'v', '1', 0};

static void cfg_fields(const gpt2_config& c, int32_t f[10]) {
    f[0] = c.n_layer; f[1] = c.n_head; f[2] = c.d_model; f[3] = c.vocab_size; f[4] = c.padded_vocab;
    f[5] = c.block_size; f[6] = c.batch_size; f[7] = c.seq_len; f[8] = c.grad_accum_steps;
    f[9] = c.precision;
}

int gpt2_save(gpt2_model* m, const char* path) {
    if (!m || !path) return GPT2_EINVAL;
    if (int r0 = join_side(m)) return r0;
    CK(m, cudaStreamSynchronize(m->stream));
    DevState st;
    CK(m, cudaMemcpy(&st, m->st, sizeof st, cudaMemcpyDeviceToHost));
    FILE* f = std::fopen(path, "wb");
    if (!f) return fail(m, GPT2_EINVAL, std::string("cannot create checkpoint file ") + path);
    int32_t fields[10];
    cfg_fields(m->cfg, fields);
    const int64_t n = m->n_arena;
    const int32_t t = st.step_t;
    bool ok = std::fwrite(CKPT_MAGIC, 1, 16, f) == 16 && std::fwrite(fields, 4, 10, f) == 10 &&
              std::fwrite(&n, 8, 1, f) == 1 && std::fwrite(&t, 4, 1, f) == 1;
    std::vector<float> host;
    try {
        host.resize((size_t)n);
    } catch (...) {
        std::fclose(f);
        return fail(m, GPT2_ENOMEM, "host buffer for the checkpoint");
    }
    const float* bufs[3] = {m->params, m->adam_m, m->adam_v};
    for (int b = 0; b < 3 && ok; b++) {
        cudaError_t e = cudaMemcpy(host.data(), bufs[b], (size_t)n * 4, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) {
            std::fclose(f);
            return fail_cuda(m, "checkpoint read-back", e);
        }
        ok = std::fwrite(host.data(), 4, (size_t)n, f) == (size_t)n;
    }
    ok = (std::fclose(f) == 0) && ok;
    if (!ok) return fail(m, GPT2_EINVAL, std::string("cannot write checkpoint file ") + path);
    return GPT2_OK;
}

int gpt2_load(gpt2_model* m, const char* path) {
    if (!m || !path) return GPT2_EINVAL;
    if (int r0 = join_side(m)) return r0;
    m->kv_len = 0;
    FILE* f = std::fopen(path, "rb");
    if (!f) return fail(m, GPT2_EINVAL, std::string("cannot open checkpoint file ") + path);
    char magic[16];
    int32_t fields[10], mine[10];
    int64_t n = 0;
    int32_t t = 0;
    bool ok = std::fread(magic, 1, 16, f) == 16 && std::memcmp(magic, CKPT_MAGIC, 16) == 0 &&
              std::fread(fields, 4, 10, f) == 10 && std::fread(&n, 8, 1, f) == 1 &&
              std::fread(&t, 4, 1, f) == 1;
    cfg_fields(m->cfg, mine);
    if (!ok || std::memcmp(fields, mine, sizeof mine) != 0 || n != m->n_arena || t < 0) {
        std::fclose(f);
        return fail(m, GPT2_EINVAL, std::string("not a checkpoint of this model configuration: ") + path);
    }
    std::vector<float> host;
    try {
        host.resize((size_t)n);
    } catch (...) {
        std::fclose(f);
        return fail(m, GPT2_ENOMEM, "host buffer for the checkpoint");
    }
    CK(m, cudaStreamSynchronize(m->stream));
    float* bufs[3] = {m->params, m->adam_m, m->adam_v};
    for (int b = 0; b < 3; b++) {
        if (std::fread(host.data(), 4, (size_t)n, f) != (size_t)n) {
            std::fclose(f);
            return fail(m, GPT2_EINVAL, std::string("truncated checkpoint file ") + path);
        }
        cudaError_t e = cudaMemcpy(bufs[b], host.data(), (size_t)n * 4, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            std::fclose(f);
            return fail_cuda(m, "checkpoint upload", e);
        }
    }
    std::fclose(f);
    CK(m, cudaMemcpy((char*)m->st + offsetof(DevState, step_t), &t, sizeof t, cudaMemcpyHostToDevice));
    if (m->use_bf16) CK(m, k::f32_to_bf16(m->params, m->pbf, m->decay_end, m->stream));
    CK(m, cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

int64_t gpt2_num_params(const gpt2_model* m, int include_wpe, int padded) {
    if (!m) return GPT2_EINVAL;
    int64_t n = 0;
    for (const auto& r : m->tensors) {
        if (r.name == "wpe" && !include_wpe) continue;
        if (r.name == "wte" && !padded) { n += (int64_t)m->V * m->C; continue; }
        n += r.numel;
    }
    return n;
}

int gpt2_host_init_tensor(const gpt2_config* cfg, uint64_t seed, int kidx, float* dst) {
    std::string why;
    int r = validate_cfg(cfg, why);
    if (r) return fail(nullptr, r, why);
    Plan p = make_plan(cfg);
    if (!dst || kidx < 0 || kidx >= (int)p.t.size()) return fail(nullptr, GPT2_EINVAL, "bad tensor index");
    host_init_tensor(cfg, p.t[kidx], kidx, seed, dst);
    return GPT2_OK;
}

int gpt2_profile(gpt2_model* m, int on) {
    if (!m) return GPT2_EINVAL;
    if (int r0 = join_side(m)) return r0;
    int r = prof_collect(m);
    if (r) return r;
    m->sites.clear();
    m->prof_on = on != 0;
    return GPT2_OK;
}

int gpt2_profile_count(gpt2_model* m) {
    if (!m) return GPT2_EINVAL;
    if (int r0 = join_side(m)) return r0;
    int r = prof_collect(m);
    if (r) return r;
    return (int)m->sites.size();
}

int gpt2_profile_entry(gpt2_model* m, int i, const char** name, int64_t* calls, int64_t* kernels,
                       double* ms, double* flops, double* bytes) {
    if (!m || i < 0 || i >= (int)m->sites.size()) return GPT2_EINVAL;
    const auto& a = m->sites[i];
    if (name) *name = a.name;
    if (calls) *calls = a.calls;
    if (kernels) *kernels = a.kernels;
    if (ms) *ms = a.ms;
    if (flops) *flops = a.flops;
    if (bytes) *bytes = a.bytes;
    return GPT2_OK;
}

// ------------------------------------------------------------------ op-level
}  // extern "C"

// Status words of the op-level calls: bounded-wait expiries inside their
// kernels are recorded in a DevState on the device the call ran on. The
// allocating entry points use one word per device, allocated on first use;
// the allocation-free attention backward uses a word compiled into the
// library (below), so that neither it nor gpt2_op_sync has to allocate.
namespace {

constexpr int OP_MAX_DEVICES = 64;
std::mutex g_op_mu;
DevState* g_op_state[OP_MAX_DEVICES] = {};

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev >= 0 && dev < OP_MAX_DEVICES ? dev : -1;
}

// The current device's status word of the allocating op-level calls, created
// (cudaMalloc) when `create` and it does not exist yet; nullptr otherwise.
DevState* op_state_dev(bool create) {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lock(g_op_mu);
    if (!g_op_state[dev] && create) {
        DevState* st = nullptr;
        if (cudaMalloc(&st, sizeof(DevState)) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        if (cudaMemset(st, 0, sizeof(DevState)) != cudaSuccess) {
            cudaFree(st);
            return nullptr;
        }
        g_op_state[dev] = st;
    }
    return g_op_state[dev];
}
DevState* op_state() { return op_state_dev(true); }

// ---------------- the allocation-free attention backward's fixed device memory
// Its rowsum scratch and its status word are file-scope device arrays: every
// device that loads this library holds them until the process exits. Host code
// must not use their names as addresses (on the host they are stand-in
// symbols), so each device's addresses are looked up once, with that device
// current, by cudaGetSymbolAddress.
constexpr int64_t NOALLOC_ROWS_MAX = int64_t(1) << 20;   // B*H*T rows, 4 MiB of fp32
__device__ __align__(256) float g_noalloc_rowsum[NOALLOC_ROWS_MAX];
__device__ __align__(256) DevState g_noalloc_state;       // zero at load

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[OP_MAX_DEVICES] = {};
DevState* g_noalloc_st[OP_MAX_DEVICES] = {};

// Device addresses of g_noalloc_rowsum and g_noalloc_state on the current
// device (looked up on the first call made on it; nothing is allocated).
cudaError_t noalloc_scratch(float** out, DevState** st) {
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        void* q = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_rowsum);
        if (e != cudaSuccess) return e;
        e = cudaGetSymbolAddress(&q, g_noalloc_state);
        if (e != cudaSuccess) return e;
        g_noalloc_st[dev] = (DevState*)q;
        g_noalloc_ptr[dev] = (float*)p;
    }
    *out = g_noalloc_ptr[dev];
    *st = g_noalloc_st[dev];
    return cudaSuccess;
}
// The no-alloc status word of the current device if the allocation-free
// entry point has run on it, else nullptr.
DevState* noalloc_state_if_used() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    return g_noalloc_st[dev];
}

// Read a status word's error bits and clear them (the wait limit stays).
cudaError_t take_status(DevState* st, unsigned int* err, unsigned int* site) {
    DevState h;
    cudaError_t r = cudaMemcpy(&h, st, sizeof h, cudaMemcpyDeviceToHost);
    if (r != cudaSuccess) return r;
    *err = h.err;
    *site = h.timeout_site;
    if (h.err) r = cudaMemset((char*)st + offsetof(DevState, err), 0, sizeof(unsigned int));
    return r;
}

}  // namespace

extern "C" {

int gpt2_op_gemm_bf16(int M, int N, int K, const void* A, int64_t lda, int a_kmajor, const void* B,
                      int64_t ldb, int b_kmajor, const float* bias, void* out_bf16, float* out_f32,
                      int64_t ldd, int accumulate, void* stream) {
    if (!A || !B || (!out_bf16 && !out_f32)) return fail(nullptr, GPT2_EINVAL, "NULL operand");
    GemmEpi e{};
    if (out_bf16) {
        e = GemmEpi{EPI_STORE_ACT, bias, out_bf16, ldd, nullptr, 0, nullptr, 0};
    } else if (accumulate) {
        if (bias) return fail(nullptr, GPT2_EINVAL, "bias with accumulate is not supported");
        e = GemmEpi{EPI_ACCUM_F32, nullptr, out_f32, ldd, nullptr, 0, nullptr, 0};
    } else {
        e = GemmEpi{EPI_STORE_F32, bias, out_f32, ldd, nullptr, 0, nullptr, 0};
    }
    GemmOperand a{A, lda, a_kmajor != 0}, b{B, ldb, b_kmajor != 0};
    if (!k::gemm_bf16_tc_supported(M, N, K, a, b, e))
        return fail(nullptr, GPT2_EINVAL, "unsupported GEMM shape/alignment");
    DevState* st = op_state();
    if (!st) return fail(nullptr, GPT2_ENOMEM, "status word allocation failed");
    cudaError_t r = k::gemm_bf16_tc(M, N, K, a, b, e, 1, st, (cudaStream_t)stream);
    if (r != cudaSuccess) return fail_cuda(nullptr, "gemm_bf16_tc", r);
    return GPT2_OK;
}

int gpt2_op_gemm_bf16_gelu(int M, int N, int K, const void* A, int64_t lda, int a_kmajor,
                           const void* B, int64_t ldb, int b_kmajor, const float* bias,
                           int backward, void* out, void* out2_or_aux, int64_t ldd, void* stream) {
    if (!A || !B || !out || !out2_or_aux) return fail(nullptr, GPT2_EINVAL, "NULL operand");
    GemmEpi e{};
    if (backward) {
        if (bias) return fail(nullptr, GPT2_EINVAL, "bias with the GELU backward epilogue");
        e = GemmEpi{EPI_GELU_BWD, nullptr, out, ldd, nullptr, 0, out2_or_aux, ldd};
    } else {
        e = GemmEpi{EPI_GELU, bias, out, ldd, out2_or_aux, ldd, nullptr, 0};
    }
    GemmOperand a{A, lda, a_kmajor != 0}, b{B, ldb, b_kmajor != 0};
    if (!k::gemm_bf16_tc_supported(M, N, K, a, b, e))
        return fail(nullptr, GPT2_EINVAL, "unsupported GEMM shape/alignment");
    DevState* st = op_state();
    if (!st) return fail(nullptr, GPT2_ENOMEM, "status word allocation failed");
    cudaError_t r = k::gemm_bf16_tc(M, N, K, a, b, e, 1, st, (cudaStream_t)stream);
    if (r != cudaSuccess) return fail_cuda(nullptr, "gemm_bf16_tc", r);
    return GPT2_OK;
}

int gpt2_op_sync(void* stream) {
    cudaError_t r = cudaStreamSynchronize((cudaStream_t)stream);
    if (r != cudaSuccess) return fail_cuda(nullptr, "cudaStreamSynchronize", r);
    // both status words of the current device; neither is created here, so
    // this call allocates nothing
    unsigned int err = 0, site = 0;
    DevState* words[2] = {op_state_dev(false), noalloc_state_if_used()};
    for (DevState* w : words) {
        if (!w) continue;
        unsigned int e = 0, s = 0;
        r = take_status(w, &e, &s);
        if (r != cudaSuccess) return fail_cuda(nullptr, "status read", r);
        if (e && !err) site = s;
        err |= e;
    }
    if (err & ERR_TIMEOUT)
        return fail(nullptr, GPT2_ETIMEOUT,
                    "a bounded device wait expired in an op-level call (site " +
                        std::to_string(site) + ")");
    return GPT2_OK;
}

int gpt2_op_set_wait_limit(unsigned int cycles) {
    // testing hook: the allocating entry points' status word (created here if
    // needed) and the allocation-free one of the current device
    DevState* st = op_state();
    if (!st) return fail(nullptr, GPT2_ENOMEM, "status word allocation failed");
    float* scratch = nullptr;
    DevState* nst = nullptr;
    cudaError_t r = noalloc_scratch(&scratch, &nst);
    if (r != cudaSuccess) return fail_cuda(nullptr, "cudaGetSymbolAddress", r);
    for (DevState* w : {st, nst}) {
        r = cudaMemcpy((char*)w + offsetof(DevState, wait_limit), &cycles, sizeof cycles,
                       cudaMemcpyHostToDevice);
        if (r != cudaSuccess) return fail_cuda(nullptr, "wait limit write", r);
    }
    return GPT2_OK;
}

int gpt2_op_sample(const float* logits, int rows, int V, int64_t ld, float temperature, int top_k,
                   const float* u, int32_t* out, int32_t* ctx, int T, int t, void* stream) {
    if (!logits || !u || !out || rows <= 0 || V <= 0 || ld < V)
        return fail(nullptr, GPT2_EINVAL, "bad sampling arguments");
    if (ctx && (T < 1 || T > 1024 || t < 1 || t > T))
        return fail(nullptr, GPT2_EINVAL, "context must have 1 <= t <= T <= 1024");
    cudaError_t r = k::sample(logits, rows, V, ld, temperature, top_k, u, out, ctx, T, t,
                              (cudaStream_t)stream);
    if (r != cudaSuccess) return fail_cuda(nullptr, "sample", r);
    return GPT2_OK;
}

int gpt2_op_attention_fwd(int precision, int B, int T, int H, int hs, const void* qkv, void* out,
                          float* lse, void* stream) {
    if (!qkv || !out || !lse || B <= 0 || T <= 0 || H <= 0 || hs <= 0)
        return fail(nullptr, GPT2_EINVAL, "bad attention arguments");
    cudaError_t r;
    if (precision == GPT2_BF16) {
        DevState* st = op_state();
        if (!st) return fail(nullptr, GPT2_ENOMEM, "status word allocation failed");
        r = k::attention_fwd_bf16((const bf16*)qkv, (bf16*)out, lse, B, T, H, hs, st,
                                  (cudaStream_t)stream);
    }
    else
        r = k::attention_fwd_f32((const float*)qkv, (float*)out, lse, B, T, H, hs, (cudaStream_t)stream);
    if (r == cudaErrorInvalidValue) return fail(nullptr, GPT2_EINVAL, "unsupported attention shape");
    if (r != cudaSuccess) return fail_cuda(nullptr, "attention_fwd", r);
    return GPT2_OK;
}

int gpt2_op_attention_bwd(int precision, int B, int T, int H, int hs, const void* qkv,
                          const void* out, const float* lse, const void* dout, void* dqkv,
                          float* scratch, void* stream) {
    if (!qkv || !out || !lse || !dout || !dqkv || !scratch || B <= 0 || T <= 0 || H <= 0 || hs <= 0)
        return fail(nullptr, GPT2_EINVAL, "bad attention arguments");
    cudaError_t r;
    if (precision == GPT2_BF16) {
        DevState* st = op_state();
        if (!st) return fail(nullptr, GPT2_ENOMEM, "status word allocation failed");
        r = k::attention_bwd_bf16((const bf16*)qkv, (const bf16*)out, lse, (const bf16*)dout,
                                  (bf16*)dqkv, scratch, B, T, H, hs, st, (cudaStream_t)stream);
    } else {
        r = k::attention_bwd_f32((const float*)qkv, (const float*)out, lse, (const float*)dout,
                                 (float*)dqkv, scratch, B, T, H, hs, (cudaStream_t)stream);
    }
    if (r == cudaErrorInvalidValue) return fail(nullptr, GPT2_EINVAL, "unsupported attention shape");
    if (r != cudaSuccess) return fail_cuda(nullptr, "attention_bwd", r);
    return GPT2_OK;
}

}  // extern "C"

// ------------------------------------------------------- allocation-free variant
// gpt2_op_attention_bwd_noalloc: the attention backward with its rowsum
// scratch in the fixed, file-scope device array above instead of a caller
// buffer, for callers that cannot allocate device memory (a plugin inside a
// host that owns the allocator and forbids cudaMalloc, code that runs while an
// allocator is locked, or a host with a hard no-allocation policy after
// start-up). Its kernels' bounded-wait expiries go to the fixed status word
// g_noalloc_state, which gpt2_op_sync reads.
extern "C" int gpt2_op_attention_bwd_noalloc(int precision, int B, int T, int H, int hs,
                                             const void* qkv, const void* out, const float* lse,
                                             const void* dout, void* dqkv, void* stream) {
    if (!qkv || !out || !lse || !dout || !dqkv || B <= 0 || T <= 0 || H <= 0 || hs <= 0)
        return fail(nullptr, GPT2_EINVAL, "bad attention arguments");
    if ((int64_t)B * H * T > NOALLOC_ROWS_MAX)
        return fail(nullptr, GPT2_EINVAL,
                    "B*H*T = " + std::to_string((int64_t)B * H * T) +
                        " exceeds the fixed scratch of the allocation-free attention backward (" +
                        std::to_string(NOALLOC_ROWS_MAX) + " rows)");
    float* scratch = nullptr;
    DevState* st = nullptr;
    cudaError_t r = noalloc_scratch(&scratch, &st);
    if (r != cudaSuccess) return fail_cuda(nullptr, "cudaGetSymbolAddress", r);
    // every row of the scratch is written by the rowsum pass before any read,
    // so stale contents from an earlier call need no clearing
    if (precision == GPT2_BF16)
        r = k::attention_bwd_bf16((const bf16*)qkv, (const bf16*)out, lse, (const bf16*)dout,
                                  (bf16*)dqkv, scratch, B, T, H, hs, st, (cudaStream_t)stream);
    else
        r = k::attention_bwd_f32((const float*)qkv, (const float*)out, lse, (const float*)dout,
                                 (float*)dqkv, scratch, B, T, H, hs, (cudaStream_t)stream);
    if (r == cudaErrorInvalidValue) return fail(nullptr, GPT2_EINVAL, "unsupported attention shape");
    if (r != cudaSuccess) return fail_cuda(nullptr, "attention_bwd_noalloc", r);
    return GPT2_OK;
}
