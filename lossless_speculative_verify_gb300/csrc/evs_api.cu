// C-ABI entry points: configuration checks, workspace layout, pass orchestration,
// state import / export. Everything is enqueued on the handle's stream; nothing here
// synchronises except evs_export_state and evs_device_flags, which say so.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "evs_internal.h"

namespace evs {

// Event pairs around launches, grouped by kernel kind (evs_profile_*).
struct Profiler {
    struct Rec { int kind; cudaEvent_t a, b; };
    std::vector<Rec> recs;
    std::vector<cudaEvent_t> pool;
    cudaEvent_t open = nullptr;
    cudaEvent_t get() {
        if (!pool.empty()) {
            cudaEvent_t e = pool.back();
            pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        cudaEventCreate(&e);
        return e;
    }
    ~Profiler() {
        for (auto& r : recs) { cudaEventDestroy(r.a); cudaEventDestroy(r.b); }
        for (auto e : pool) cudaEventDestroy(e);
        if (open) cudaEventDestroy(open);
    }
};

// Inside stream capture a plain record only orders streams; an external record becomes an
// event node of the graph, which is what timing needs.
static void record(cudaEvent_t e, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cs);
    if (cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
    else
        cudaEventRecord(e, s);
}

void prof_begin(evs_handle* h, int kind) {
    (void)kind;
    if (!h->prof_on) return;
    Profiler* p = (Profiler*)h->prof;
    p->open = p->get();
    record(p->open, h->stream);
}

void prof_end(evs_handle* h, int kind) {
    if (!h->prof_on) return;
    Profiler* p = (Profiler*)h->prof;
    cudaEvent_t e = p->get();
    record(e, h->stream);
    p->recs.push_back({kind, p->open, e});
    p->open = nullptr;
}

}  // namespace evs

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

inline int elem_bytes(const evs_config& c) { return c.dtype == EVS_DTYPE_BF16 ? 2 : 4; }

bool valid_config(const evs_config* c) {
    if (!c) return false;
    if (c->d < 64 || c->d > 8192 || c->d % 64) return false;
    if (!(c->vocab == 256 || c->vocab == 512 || c->vocab == 1024 || c->vocab == 2048 || c->vocab == 4096))
        return false;
    if (c->n_layers < 1 || c->n_layers > EVS_MAX_LAYERS) return false;
    if (!(c->head_dim == 16 || c->head_dim == 32 || c->head_dim == 64 || c->head_dim == 128)) return false;
    for (int i = 0; i < c->n_layers; ++i) {
        const int k = c->layer_kind[i], p = c->layer_param[i];
        if (k == EVS_LAYER_FIR) {
            if (p < 2 || p > 16) return false;
        } else if (k == EVS_LAYER_IIR) {
            if (!(p == 1 || p == 2 || p == 4 || p == 8 || p == 16 || p == 32)) return false;
        } else if (k == EVS_LAYER_ATTN) {
            if (p < 1 || (long long)p * c->head_dim != c->d) return false;
        } else {
            return false;
        }
    }
    if (c->gamma < 1 || c->gamma > 31) return false;
    if (c->batch < 1 || c->batch > 64 || c->n_cand < 1 || c->n_cand > 16) return false;
    if ((long long)c->batch * c->n_cand * (c->gamma + 1) > 512) return false;
    if (c->prefill_chunk < 1 || c->prefill_chunk > 128) return false;
    if ((long long)c->batch * c->prefill_chunk > 512) return false;
    if (c->t_max < 1 || c->t_max > (1 << 21)) return false;
    if (c->dtype != EVS_DTYPE_F32 && c->dtype != EVS_DTYPE_BF16) return false;
    if (c->mode != EVS_MODE_GREEDY && c->mode != EVS_MODE_SAMPLING) return false;
    if (c->cand_rule != EVS_CAND_RECURSIVE && c->cand_rule != EVS_CAND_MAX_ACCEPT) return false;
    if (!(c->temperature > 0.f) || !(c->near_tie_tau >= 0.f)) return false;
    return true;
}

evs::Geometry geometry(const evs_config& c) {
    evs::Geometry g{};
    g.B = c.batch;
    g.C = c.n_cand;
    g.T = c.gamma + 1;
    g.M_verify = g.B * g.C * g.T;
    g.M_max = std::max(g.M_verify, g.B * c.prefill_chunk);
    g.q_max = std::max(g.C * g.T, c.prefill_chunk);
    g.h_max = 1;
    for (int i = 0; i < c.n_layers; ++i)
        if (c.layer_kind[i] == EVS_LAYER_ATTN) g.h_max = std::max(g.h_max, c.layer_param[i]);
    // prefix split so that splits x sequences x heads covers the 152 SMs about four times
    const long long target = std::max(1LL, (4LL * 152 + (long long)g.B * g.h_max - 1) / ((long long)g.B * g.h_max));
    long long chunk = (c.t_max + target - 1) / target;
    chunk = std::max(64LL, (chunk + 63) / 64 * 64);
    g.kv_chunk = (int)chunk;
    g.kv_splits = (int)((c.t_max + chunk - 1) / chunk);
    return g;
}

// Lays out every buffer inside the workspace starting at base (or at 0 to size it).
size_t carve(const evs_config& c, char* base, evs_handle* h) {
    const evs::Geometry g = geometry(c);
    const size_t es = elem_bytes(c);
    const size_t B = c.batch, C = c.n_cand, T = g.T, d = c.d, dh = c.head_dim;
    size_t off = 0;
    auto take = [&](size_t bytes) -> char* {
        char* p = base ? base + off : nullptr;
        off = align_up(off + bytes);
        return p;
    };
    char* kv_len = take(B * 4);
    char* kv_base = take(B * 4);
    char* flags = take(4);
    char* cand_k = take(B * C * 4);
    char* cand_corr = take(B * C * 4);
    char* cand_tie = take(B * C * 4);
    char* layer_dev = take(sizeof(evs::LayerDesc) * c.n_layers);
    if (h) {
        h->kv_len = (int32_t*)kv_len;
        h->kv_base = (int32_t*)kv_base;
        h->flags = (uint32_t*)flags;
        h->cand_k = (int32_t*)cand_k;
        h->cand_corr = (int32_t*)cand_corr;
        h->cand_tie = (uint32_t*)cand_tie;
        h->layer_dev = (evs::LayerDesc*)layer_dev;
    }
    for (int i = 0; i < c.n_layers; ++i) {
        evs::LayerDesc L{};
        L.kind = c.layer_kind[i];
        L.param = c.layer_param[i];
        size_t tail_b = 0, stage_b = 0, state_b = 0, uin_b = 0, cache_b = 0, side_b = 0;
        if (L.kind == EVS_LAYER_FIR) {
            tail_b = B * (L.param - 1) * d * 4;
            stage_b = B * C * (L.param - 1 + T) * d * 4;
            L.tail = (float*)take(tail_b);
            L.stage = (float*)take(stage_b);
        } else if (L.kind == EVS_LAYER_IIR) {
            state_b = B * d * L.param * 8;
            uin_b = B * C * T * d * 4;
            L.state = (float2*)take(state_b);
            L.uin = (float*)take(uin_b);
            if (h) {
                L.lam = (const float2*)h->w.layer[i].iir_lambda;
                L.bq = (const float2*)h->w.layer[i].iir_b;
            }
        } else {
            cache_b = B * (size_t)L.param * (size_t)c.t_max * dh * es;
            L.kc = take(cache_b);
            L.vc = take(cache_b);
            if (C > 1) {
                side_b = B * C * (size_t)L.param * T * dh * es;
                L.ks = take(side_b);
                L.vs = take(side_b);
            }
        }
        if (h) {
            h->layer[i] = L;
            h->tail_bytes[i] = tail_b;
            h->stage_bytes[i] = stage_b;
            h->state_bytes[i] = state_b;
            h->uin_bytes[i] = uin_b;
            h->cache_bytes[i] = cache_b;
            h->side_bytes[i] = side_b;
        }
    }
    char* hbuf = take((size_t)g.M_max * d * 4);
    char* hb = take((size_t)g.M_max * d * 2);
    char* ssq = take((size_t)(d / 128 + 1) * g.M_max * 4);
    char* act = take((size_t)g.M_max * d * es);
    char* y = take((size_t)g.M_max * 3 * d * 4);
    char* logits = take((size_t)g.M_verify * c.vocab * 4);
    size_t splits_max = g.kv_splits;
    if (c.dtype == EVS_DTYPE_BF16 && c.head_dim == 128) {
        // the tensor-core attention may chunk the prefix more finely (its plan depends only
        // on the pass shape and t_max; 200 KiB stands in for the shared-memory limit here)
        const evs::AttnPlan pv = evs::attn_plan(g.C * g.T, g.B, g.h_max, c.t_max, 200 * 1024);
        const evs::AttnPlan pp = evs::attn_plan(c.prefill_chunk, g.B, g.h_max, c.t_max, 200 * 1024);
        splits_max = std::max(splits_max, (size_t)std::max(pv.splits, pp.splits));
    }
    char* part = take(B * (size_t)g.h_max * splits_max * g.q_max * (dh + 2) * 4);
    // split-K partials: splits x tiles <= the CTA target, so splits x N <= target x 128
    const size_t gpart_floats = (size_t)evs::tc_cta_target() * 128 * g.M_max;
    char* gpart = take(gpart_floats * 4);
    char* gcnt = take((size_t)(std::max(3 * c.d, c.vocab) / 128 + 1) * 4);
    if (h) {
        h->h = (float*)hbuf;
        h->hb = (__nv_bfloat16*)hb;
        h->ssq = (float*)ssq;
        h->act = act;
        h->y = (float*)y;
        h->logits = (float*)logits;
        h->attn_part = (float*)part;
        h->gemm_part = (float*)gpart;
        h->gemm_part_floats = gpart_floats;
        h->gemm_counters = (int*)gcnt;
        h->g = g;
    }
    return off;
}

evs_status cuda_ok(cudaError_t e) { return e == cudaSuccess ? EVS_OK : EVS_ERR_CUDA; }

evs_status after_launch(evs_handle* h) {
    (void)h;
    return cuda_ok(cudaGetLastError());
}

bool weights_ok(const evs_config& c, const evs_weights* w) {
    if (!w || !w->embed || !w->head) return false;
    for (int i = 0; i < c.n_layers; ++i) {
        const evs_layer_weights& L = w->layer[i];
        switch (c.layer_kind[i]) {
            case EVS_LAYER_FIR:
                if (!L.w_in || !L.w_out || !L.fir_taps) return false;
                break;
            case EVS_LAYER_IIR:
                if (!L.w_in || !L.w_out || !L.iir_lambda || !L.iir_b || !L.iir_c) return false;
                break;
            default:
                if (!L.w_qkv || !L.w_o) return false;
        }
    }
    return true;
}

evs_status zero_state(evs_handle* h) {
    const evs_config& c = h->cfg;
    cudaStream_t s = h->stream;
    if (cudaMemsetAsync(h->kv_len, 0, c.batch * 4, s) != cudaSuccess) return EVS_ERR_CUDA;
    if (cudaMemsetAsync(h->kv_base, 0, c.batch * 4, s) != cudaSuccess) return EVS_ERR_CUDA;
    for (int i = 0; i < c.n_layers; ++i) {
        const evs::LayerDesc& L = h->layer[i];
        if (L.kind == EVS_LAYER_FIR && cudaMemsetAsync(L.tail, 0, h->tail_bytes[i], s) != cudaSuccess)
            return EVS_ERR_CUDA;
        if (L.kind == EVS_LAYER_IIR && cudaMemsetAsync(L.state, 0, h->state_bytes[i], s) != cudaSuccess)
            return EVS_ERR_CUDA;
    }
    h->kv_hi = 0;
    h->verified = 0;
    return EVS_OK;
}

// Where a layer's in-projection leaves the mixer input: a verify pass keeps an IIR layer's
// scan inputs u_0..u_gamma in the layer's own buffer, from which slicing recomputes s_k;
// everything else goes through the shared projection output.
float* mixer_input(evs_handle* h, int li, const evs::Pass& p) {
    return h->cfg.layer_kind[li] == EVS_LAYER_IIR && !p.commit ? h->layer[li].uin : h->y;
}

// One block pass through every layer (Lemma 2: a single forward from the pre-round state).
void run_layers(evs_handle* h, const int32_t* tokens, int tok_stride, const int32_t* anchor,
                const evs::Pass& p, bool with_head) {
    const evs_config& c = h->cfg;
    const int d = c.d;
    evs::launch_embed(h, tokens, tok_stride, anchor, p);
    if (h->fused) {
        // RMS norm folded into the projections: consumers of h read bf16(h) and scale their
        // output rows by 1/rms(h); producers of h leave bf16(h) and per-tile sums of squares
        const evs::GemmFuse in{h->ssq, d / 128, h->g.M_max, d, nullptr, 0, nullptr, -1, -1, &p};
        const evs::GemmFuse out{nullptr, 0, h->g.M_max, d, h->hb, d, h->ssq, -1, -1, &p};
        for (int li = 0; li < c.n_layers; ++li) {
            const evs_layer_weights& W = h->w.layer[li];
            int fused = 0;
            evs::GemmFuse mixin = in;
            switch (c.layer_kind[li]) {
                case EVS_LAYER_FIR:
                case EVS_LAYER_IIR: {
                    // the mixer runs in the in-projection's epilogue when the shape allows
                    mixin.mix_layer = h->fuse_mixer ? li : -1;
                    float* v = mixer_input(h, li, p);
                    const int ldv = v == h->y ? 3 * d : d;
                    evs::launch_gemm(h, h->hb, W.w_in, v, p.M, d, d, ldv, 0, &mixin, &fused);
                    if (!(fused & 1)) {
                        if (c.layer_kind[li] == EVS_LAYER_FIR)
                            evs::launch_fir(h, li, p);
                        else
                            evs::launch_iir(h, li, p, v, ldv);
                    }
                    evs::launch_gemm(h, h->act, W.w_out, h->h, p.M, d, d, d, 1, &out);
                    break;
                }
                default:
                    mixin.kv_layer = li;   // K/V rows written straight from the QKV epilogue
                    evs::launch_gemm(h, h->hb, W.w_qkv, h->y, p.M, 3 * d, d, 3 * d, 0, &mixin, &fused);
                    if (!(fused & 2)) evs::launch_kv_write(h, li, p);
                    evs::launch_attention(h, li, p);
                    evs::launch_gemm(h, h->act, W.w_o, h->h, p.M, d, d, d, 1, &out);
            }
        }
        if (with_head) evs::launch_gemm(h, h->hb, h->w.head, h->logits, p.M, c.vocab, d, c.vocab, 0, &in);
        return;
    }
    for (int li = 0; li < c.n_layers; ++li) {
        const evs_layer_weights& W = h->w.layer[li];
        evs::launch_rmsnorm(h, p);
        switch (c.layer_kind[li]) {
            case EVS_LAYER_FIR:
                evs::launch_gemm(h, h->act, W.w_in, h->y, p.M, d, d, 3 * d, 0);
                evs::launch_fir(h, li, p);
                evs::launch_gemm(h, h->act, W.w_out, h->h, p.M, d, d, d, 1);
                break;
            case EVS_LAYER_IIR: {
                float* v = mixer_input(h, li, p);
                const int ldv = v == h->y ? 3 * d : d;
                evs::launch_gemm(h, h->act, W.w_in, v, p.M, d, d, ldv, 0);
                evs::launch_iir(h, li, p, v, ldv);
                evs::launch_gemm(h, h->act, W.w_out, h->h, p.M, d, d, d, 1);
                break;
            }
            default:
                evs::launch_gemm(h, h->act, W.w_qkv, h->y, p.M, 3 * d, d, 3 * d, 0);
                evs::launch_kv_write(h, li, p);
                evs::launch_attention(h, li, p);
                evs::launch_gemm(h, h->act, W.w_o, h->h, p.M, d, d, d, 1);
        }
    }
    if (with_head) {
        evs::launch_rmsnorm(h, p);
        evs::launch_gemm(h, h->act, h->w.head, h->logits, p.M, c.vocab, d, c.vocab, 0);
    }
}

}  // namespace

extern "C" {

size_t evs_workspace_bytes(const evs_config* cfg) {
    if (!valid_config(cfg)) return 0;
    return carve(*cfg, nullptr, nullptr);
}

evs_status evs_create(const evs_config* cfg, const evs_weights* weights, void* workspace, size_t ws_bytes,
                      void* stream, evs_handle** out) {
    if (!out) return EVS_ERR_INVALID_ARG;
    *out = nullptr;
    if (!valid_config(cfg) || !weights_ok(*cfg, weights) || !workspace) return EVS_ERR_INVALID_ARG;
    if ((uintptr_t)workspace % kAlign) return EVS_ERR_INVALID_ARG;
    const size_t need = carve(*cfg, nullptr, nullptr);
    if (ws_bytes < need) return EVS_ERR_CAPACITY;
    evs_handle* h = (evs_handle*)calloc(1, sizeof(evs_handle));
    if (!h) return EVS_ERR_INVALID_ARG;
    h->cfg = *cfg;
    h->w = *weights;
    h->stream = (cudaStream_t)stream;
    h->ws = (char*)workspace;
    h->ws_bytes = ws_bytes;
    carve(*cfg, h->ws, h);
    h->tc_smem_max = 0;
    h->pdl = 1;
    h->fuse_mixer = 1;
    // the norm is folded into the tensor-core projections when every projection shape runs
    // on them (bf16, widths in whole 128-channel tiles)
    h->fused = cfg->dtype == EVS_DTYPE_BF16 && cfg->d % 128 == 0 && cfg->vocab % 128 == 0 && h->g.M_max <= 512;
    if (cfg->dtype == EVS_DTYPE_BF16) {
        h->tc_smem_max = evs::gemm_tc_init();
        const int attn_smem = evs::attn_init();
        if (h->tc_smem_max < 0 || attn_smem < 0) {
            free(h);
            return EVS_ERR_CUDA;
        }
        if (cfg->head_dim == 128) {
            // plans use at most 200 KiB, the bound the partial buffer was sized with
            const int sm = std::min(attn_smem, 200 * 1024);
            h->plan_verify = evs::attn_plan(h->g.C * h->g.T, h->g.B, h->g.h_max, cfg->t_max, sm);
            h->plan_prefill = evs::attn_plan(cfg->prefill_chunk, h->g.B, h->g.h_max, cfg->t_max, sm);
        }
    }
    evs_status st = cuda_ok(cudaMemcpyAsync(h->layer_dev, h->layer, sizeof(evs::LayerDesc) * cfg->n_layers,
                                            cudaMemcpyHostToDevice, h->stream));
    if (st == EVS_OK) st = cuda_ok(cudaMemsetAsync(h->flags, 0, 4, h->stream));
    if (st == EVS_OK)
        st = cuda_ok(cudaMemsetAsync(h->gemm_counters, 0, (std::max(3 * cfg->d, cfg->vocab) / 128 + 1) * 4,
                                     h->stream));
    if (st == EVS_OK) st = zero_state(h);
    for (int i = 0; i < cfg->n_layers && st == EVS_OK; ++i) {
        // never-written cache rows are read (and multiplied by zero weights) at chunk edges
        if (h->layer[i].kind != EVS_LAYER_ATTN) continue;
        st = cuda_ok(cudaMemsetAsync(h->layer[i].kc, 0, h->cache_bytes[i], h->stream));
        if (st == EVS_OK) st = cuda_ok(cudaMemsetAsync(h->layer[i].vc, 0, h->cache_bytes[i], h->stream));
    }
    if (st == EVS_OK) st = cuda_ok(cudaStreamSynchronize(h->stream));  // layer table copied from host
    if (st != EVS_OK) {
        free(h);
        return st;
    }
    *out = h;
    return EVS_OK;
}

void evs_destroy(evs_handle* h) {
    if (!h) return;
    delete (evs::Profiler*)h->prof;
    free(h);
}

evs_status evs_profile_enable(evs_handle* h, int32_t on) {
    if (!h) return EVS_ERR_INVALID_ARG;
    if (on && !h->prof) h->prof = new evs::Profiler();
    h->prof_on = on ? 1 : 0;
    return EVS_OK;
}

evs_status evs_profile_read(evs_handle* h, int32_t* launches, float* ms, int32_t n) {
    if (!h || !launches || !ms || n < 0) return EVS_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) { launches[i] = 0; ms[i] = 0.f; }
    evs::Profiler* p = (evs::Profiler*)h->prof;
    if (!p) return EVS_OK;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return EVS_ERR_CUDA;
    for (auto& r : p->recs) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) {
            cudaGetLastError();  // not sticky: leave no error for later launches to report
            p->recs.clear();
            return EVS_ERR_CUDA;
        }
        if (r.kind >= 0 && r.kind < n) { launches[r.kind] += 1; ms[r.kind] += t; }
        p->pool.push_back(r.a);
        p->pool.push_back(r.b);
    }
    p->recs.clear();
    return EVS_OK;
}

evs_status evs_set_stream(evs_handle* h, void* stream) {
    if (!h) return EVS_ERR_INVALID_ARG;
    h->stream = (cudaStream_t)stream;
    return EVS_OK;
}

evs_status evs_reset(evs_handle* h) {
    if (!h) return EVS_ERR_INVALID_ARG;
    h->launches = 0;
    return zero_state(h);
}

evs_status evs_prefill(evs_handle* h, const int32_t* tokens, int32_t P) {
    if (!h || P < 0 || (P > 0 && !tokens)) return EVS_ERR_INVALID_ARG;
    h->launches = 0;
    if (h->kv_hi + P > h->cfg.t_max) return EVS_ERR_CAPACITY;
    const int B = h->cfg.batch, chunk = h->cfg.prefill_chunk;
    for (int off = 0; off < P; off += chunk) {
        const int T = std::min(chunk, P - off);
        evs::Pass p{B, 1, T, B * T, 1, 1};
        run_layers(h, tokens + off, P, nullptr, p, false);
        evs::launch_advance(h, T);
    }
    h->kv_hi += P;
    h->verified = 0;
    return after_launch(h);
}

evs_status evs_verify_block(evs_handle* h, const int32_t* tokens, const int32_t* anchor, const float* q_probs,
                            const float* uniforms, int32_t* accepted_len, int32_t* correction,
                            int32_t* best_cand, uint32_t* near_tie) {
    if (!h || !tokens || !accepted_len || !correction) return EVS_ERR_INVALID_ARG;
    const evs_config& c = h->cfg;
    if (c.mode == EVS_MODE_SAMPLING && (!q_probs || !uniforms)) return EVS_ERR_INVALID_ARG;
    if (c.n_cand > 1 && !best_cand) return EVS_ERR_INVALID_ARG;
    h->launches = 0;
    const int T = c.gamma + 1;
    if (h->kv_hi + T > c.t_max) return EVS_ERR_CAPACITY;
    evs::Pass p{c.batch, c.n_cand, T, h->g.M_verify, 0, c.n_cand == 1 ? 1 : 0};
    run_layers(h, tokens, T, anchor, p, true);
    evs::launch_accept(h, tokens, q_probs, uniforms, accepted_len, correction, best_cand, near_tie);
    h->verified = 1;
    return after_launch(h);
}

evs_status evs_replay_state(evs_handle* h, const int32_t* tokens, const int32_t* anchor,
                            const int32_t* accepted_len, const int32_t* best_cand) {
    if (!h || !tokens || !accepted_len) return EVS_ERR_INVALID_ARG;
    const evs_config& c = h->cfg;
    if (c.batch != 1 || (c.n_cand > 1 && !best_cand)) return EVS_ERR_INVALID_ARG;
    if (!h->verified) return EVS_ERR_STATE;
    h->launches = 0;
    int32_t kc[2] = {0, 0};
    if (cudaMemcpyAsync(&kc[0], accepted_len, 4, cudaMemcpyDeviceToHost, h->stream) != cudaSuccess ||
        (best_cand && cudaMemcpyAsync(&kc[1], best_cand, 4, cudaMemcpyDeviceToHost, h->stream) != cudaSuccess) ||
        cudaStreamSynchronize(h->stream) != cudaSuccess)
        return EVS_ERR_CUDA;
    const int k = kc[0], cand = c.n_cand > 1 ? kc[1] : 0, T = c.gamma + 1;
    if (k < 0 || k > c.gamma || cand < 0 || cand >= c.n_cand) return EVS_ERR_INVALID_ARG;
    // the accepted tokens of the candidate, consumed prefill_chunk at a time from the
    // pre-round state (the verify left the state itself untouched)
    const int32_t* acc = tokens + (size_t)cand * T;
    for (int off = 0; off <= k; off += c.prefill_chunk) {
        const int n = std::min(c.prefill_chunk, k + 1 - off);
        evs::Pass p{1, 1, n, n, 1, 1};
        run_layers(h, acc + off, T, off == 0 ? anchor : nullptr, p, false);
        evs::launch_advance(h, n);
    }
    h->kv_hi += T;
    if (h->kv_hi > c.t_max) h->kv_hi = c.t_max;
    h->verified = 0;
    return after_launch(h);
}

evs_status evs_decode_step(evs_handle* h, const int32_t* tokens, const float* uniforms, int32_t* next,
                           uint32_t* near_tie) {
    if (!h || !tokens || !next) return EVS_ERR_INVALID_ARG;
    if (h->cfg.mode == EVS_MODE_SAMPLING && !uniforms) return EVS_ERR_INVALID_ARG;
    h->launches = 0;
    if (h->kv_hi + 1 > h->cfg.t_max) return EVS_ERR_CAPACITY;
    const int B = h->cfg.batch;
    evs::Pass p{B, 1, 1, B, 1, 1};   // one committed position per sequence
    run_layers(h, tokens, 1, nullptr, p, true);
    evs::launch_advance(h, 1);
    evs::launch_pick(h, uniforms, next, near_tie);
    h->kv_hi += 1;
    h->verified = 0;
    return after_launch(h);
}

evs_status evs_slice_state(evs_handle* h, const int32_t* accepted_len, const int32_t* best_cand) {
    if (!h || !accepted_len) return EVS_ERR_INVALID_ARG;
    if (h->cfg.n_cand > 1 && !best_cand) return EVS_ERR_INVALID_ARG;
    if (!h->verified) return EVS_ERR_STATE;
    h->launches = 0;
    evs::launch_slice(h, accepted_len, best_cand);
    h->kv_hi += h->cfg.gamma + 1;
    if (h->kv_hi > h->cfg.t_max) h->kv_hi = h->cfg.t_max;
    h->verified = 0;
    return after_launch(h);
}

evs_status evs_import_state(evs_handle* h, const evs_state_view* v) {
    if (!h || !v || !v->kv_len) return EVS_ERR_INVALID_ARG;
    const evs_config& c = h->cfg;
    h->launches = 0;
    const size_t es = elem_bytes(c), dh = c.head_dim;
    long long hi = 0;
    for (int b = 0; b < c.batch; ++b) {
        const int n = v->kv_len[b];
        if (n < 0) return EVS_ERR_INVALID_ARG;
        if (n > c.t_max || n > v->t_stride) return EVS_ERR_CAPACITY;
        hi = std::max(hi, (long long)n);
    }
    for (int i = 0; i < c.n_layers; ++i) {
        const evs::LayerDesc& L = h->layer[i];
        if (L.kind == EVS_LAYER_ATTN) {
            if (!v->k[i] || !v->v[i]) return EVS_ERR_INVALID_ARG;
        } else if (L.kind == EVS_LAYER_FIR) {
            if (!v->fir_tail[i]) return EVS_ERR_INVALID_ARG;
        } else if (!v->iir_state[i]) {
            return EVS_ERR_INVALID_ARG;
        }
    }
    cudaStream_t s = h->stream;
    if (cudaMemcpyAsync(h->kv_len, v->kv_len, c.batch * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return EVS_ERR_CUDA;
    for (int i = 0; i < c.n_layers; ++i) {
        const evs::LayerDesc& L = h->layer[i];
        if (L.kind == EVS_LAYER_ATTN) {
            const size_t H = L.param;
            for (int b = 0; b < c.batch; ++b) {
                const size_t n = v->kv_len[b];
                if (!n) continue;
                const size_t dpitch = (size_t)c.t_max * dh * es, spitch = (size_t)v->t_stride * dh * es;
                char* dk = (char*)L.kc + b * H * dpitch;
                char* dv = (char*)L.vc + b * H * dpitch;
                const char* sk = (const char*)v->k[i] + b * H * spitch;
                const char* sv = (const char*)v->v[i] + b * H * spitch;
                if (cudaMemcpy2DAsync(dk, dpitch, sk, spitch, n * dh * es, H, cudaMemcpyDefault, s) != cudaSuccess ||
                    cudaMemcpy2DAsync(dv, dpitch, sv, spitch, n * dh * es, H, cudaMemcpyDefault, s) != cudaSuccess)
                    return EVS_ERR_CUDA;
            }
        } else if (L.kind == EVS_LAYER_FIR) {
            if (cudaMemcpyAsync(L.tail, v->fir_tail[i], h->tail_bytes[i], cudaMemcpyDefault, s) != cudaSuccess)
                return EVS_ERR_CUDA;
        } else {
            if (cudaMemcpyAsync(L.state, v->iir_state[i], h->state_bytes[i], cudaMemcpyDefault, s) != cudaSuccess)
                return EVS_ERR_CUDA;
        }
    }
    // the host kv_len array may be reused by the caller as soon as this returns
    if (cudaStreamSynchronize(s) != cudaSuccess) return EVS_ERR_CUDA;
    h->kv_hi = hi;
    h->verified = 0;
    return EVS_OK;
}

evs_status evs_export_state(evs_handle* h, const evs_state_view* v) {
    if (!h || !v || !v->kv_len) return EVS_ERR_INVALID_ARG;
    const evs_config& c = h->cfg;
    h->launches = 0;
    cudaStream_t s = h->stream;
    const size_t es = elem_bytes(c), dh = c.head_dim;
    if (cudaMemcpyAsync(v->kv_len, h->kv_len, c.batch * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return EVS_ERR_CUDA;
    for (int b = 0; b < c.batch; ++b)
        if (v->kv_len[b] > v->t_stride) return EVS_ERR_CAPACITY;
    for (int i = 0; i < c.n_layers; ++i) {
        const evs::LayerDesc& L = h->layer[i];
        if (L.kind == EVS_LAYER_ATTN) {
            if (!v->k[i] || !v->v[i]) continue;
            const size_t H = L.param;
            for (int b = 0; b < c.batch; ++b) {
                const size_t n = v->kv_len[b];
                if (!n) continue;
                const size_t spitch = (size_t)c.t_max * dh * es, dpitch = (size_t)v->t_stride * dh * es;
                if (cudaMemcpy2DAsync((char*)v->k[i] + b * H * dpitch, dpitch, (const char*)L.kc + b * H * spitch,
                                      spitch, n * dh * es, H, cudaMemcpyDefault, s) != cudaSuccess ||
                    cudaMemcpy2DAsync((char*)v->v[i] + b * H * dpitch, dpitch, (const char*)L.vc + b * H * spitch,
                                      spitch, n * dh * es, H, cudaMemcpyDefault, s) != cudaSuccess)
                    return EVS_ERR_CUDA;
            }
        } else if (L.kind == EVS_LAYER_FIR) {
            if (v->fir_tail[i] &&
                cudaMemcpyAsync(v->fir_tail[i], L.tail, h->tail_bytes[i], cudaMemcpyDefault, s) != cudaSuccess)
                return EVS_ERR_CUDA;
        } else if (v->iir_state[i] &&
                   cudaMemcpyAsync(v->iir_state[i], L.state, h->state_bytes[i], cudaMemcpyDefault, s) != cudaSuccess) {
            return EVS_ERR_CUDA;
        }
    }
    return cuda_ok(cudaStreamSynchronize(s));
}

evs_status evs_debug_buffer(evs_handle* h, int32_t which, int32_t layer, evs_buffer_info* out) {
    if (!h || !out) return EVS_ERR_INVALID_ARG;
    const evs_config& c = h->cfg;
    const bool per_layer = !(which == EVS_BUF_LOGITS || which == EVS_BUF_KV_LEN || which == EVS_BUF_CAND_K ||
                             which == EVS_BUF_CAND_CORR);
    if (per_layer && (layer < 0 || layer >= c.n_layers)) return EVS_ERR_INVALID_ARG;
    const evs::LayerDesc* L = per_layer ? &h->layer[layer] : nullptr;
    void* p = nullptr;
    size_t n = 0;
    switch (which) {
        case EVS_BUF_LOGITS: p = h->logits; n = (size_t)h->g.M_verify * c.vocab * 4; break;
        case EVS_BUF_KV_LEN: p = h->kv_len; n = c.batch * 4; break;
        case EVS_BUF_CAND_K: p = h->cand_k; n = (size_t)c.batch * c.n_cand * 4; break;
        case EVS_BUF_CAND_CORR: p = h->cand_corr; n = (size_t)c.batch * c.n_cand * 4; break;
        case EVS_BUF_FIR_STAGE: p = L->stage; n = h->stage_bytes[layer]; break;
        case EVS_BUF_FIR_TAIL: p = L->tail; n = h->tail_bytes[layer]; break;
        case EVS_BUF_IIR_U: p = L->uin; n = h->uin_bytes[layer]; break;
        case EVS_BUF_IIR_STATE: p = L->state; n = h->state_bytes[layer]; break;
        case EVS_BUF_K_CACHE: p = L->kc; n = h->cache_bytes[layer]; break;
        case EVS_BUF_V_CACHE: p = L->vc; n = h->cache_bytes[layer]; break;
        case EVS_BUF_K_SIDE: p = L->ks; n = h->side_bytes[layer]; break;
        case EVS_BUF_V_SIDE: p = L->vs; n = h->side_bytes[layer]; break;
        default: return EVS_ERR_INVALID_ARG;
    }
    if (!p) return EVS_ERR_INVALID_ARG;
    out->ptr = p;
    out->bytes = n;
    return EVS_OK;
}

evs_status evs_device_flags(evs_handle* h, uint32_t* flags, int32_t clear) {
    if (!h || !flags) return EVS_ERR_INVALID_ARG;
    if (cudaMemcpyAsync(flags, h->flags, 4, cudaMemcpyDeviceToHost, h->stream) != cudaSuccess) return EVS_ERR_CUDA;
    if (clear && cudaMemsetAsync(h->flags, 0, 4, h->stream) != cudaSuccess) return EVS_ERR_CUDA;
    return cuda_ok(cudaStreamSynchronize(h->stream));
}

int32_t evs_last_launch_count(evs_handle* h) { return h ? h->launches : 0; }

evs_status evs_debug_projection(evs_handle* h, const void* X, int32_t x_rows, const void* W, float* Y, int32_t M,
                                int32_t N, int32_t K, int32_t ldy, int32_t accumulate) {
    if (!h || !X || !W || !Y || h->cfg.dtype != EVS_DTYPE_BF16) return EVS_ERR_INVALID_ARG;
    if (!evs::gemm_tc_supported(M, N, K) || x_rows < M || K > h->cfg.d || ldy < N ||
        N > std::max(3 * h->cfg.d, h->cfg.vocab) || M > h->g.M_max)
        return EVS_ERR_INVALID_ARG;
    h->launches = 0;
    if (!evs::launch_gemm_tc(h, X, x_rows, W, Y, M, N, K, ldy, accumulate)) return EVS_ERR_CUDA;
    h->launches = 1;
    return after_launch(h);
}

const char* evs_status_str(evs_status s) {
    switch (s) {
        case EVS_OK: return "ok";
        case EVS_ERR_INVALID_ARG: return "invalid argument";
        case EVS_ERR_CAPACITY: return "capacity exceeded (KV rows beyond t_max or workspace too small)";
        case EVS_ERR_STATE: return "call out of order (slice without a preceding verify)";
        case EVS_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

}  // extern "C"
