// q3i8 engine: the C ABI of include/q3i8.h on one GB300 (sm_103a).
//
// Owns the device copies of the weights (repacked at init), the bf16 KV
// cache, the per-step device state (tokens, positions, step counter) and
// one captured CUDA graph per batch size for the decode step.  The decode
// loop replays that graph; next-token ids and positions stay on the device,
// so nothing crosses to the host between steps.
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <thread>
#include <vector>

#include "../../include/q3i8.h"
#include "engine.h"
#include "kernels.h"
#include "persistent.h"

using namespace q3;

static thread_local std::string g_tls_error;

static int fail(q3i8_ctx* c, int code, const char* fmt, ...) {
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (c) c->err = buf;
    else g_tls_error = buf;
    return code;
}

// Records an error of a call that has no context; q3i8_last_error(NULL)
// returns it on the same thread.
int q3_report_error(int code, const char* msg) {
    g_tls_error = msg;
    return code;
}

#define CK(c, call)                                                                                     \
    do {                                                                                                \
        cudaError_t e_ = (call);                                                                        \
        if (e_ != cudaSuccess) {                                                                        \
            int code_ = (e_ == cudaErrorMemoryAllocation) ? Q3_ERR_OOM : Q3_ERR_CUDA;                   \
            return fail((c), code_, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__,   \
                        __LINE__);                                                                      \
        }                                                                                               \
    } while (0)

// ------------------------------------------------------------------ validation

extern "C" int q3i8_validate_dims(const q3i8_dims* d, char* msg, size_t msg_cap) {
    std::string m;
    int code = Q3_OK;
    auto add = [&](int c, const std::string& s) {
        if (!m.empty()) m += "; ";
        m += s;
        if (code == Q3_OK || c == Q3_ERR_INVALID_ARGUMENTS) code = c;
    };
    if (!d) {
        add(Q3_ERR_INVALID_ARGUMENTS, "dims is NULL");
    } else {
        const int pos[] = {d->hidden, d->n_layers, d->n_heads, d->n_kv_heads, d->head_dim, d->intermediate, d->vocab};
        const char* names[] = {"hidden", "n_layers", "n_heads", "n_kv_heads", "head_dim", "intermediate", "vocab"};
        bool sizes_ok = true;
        for (int i = 0; i < 7; ++i)
            if (pos[i] <= 0) {
                add(Q3_ERR_INVALID_ARGUMENTS, std::string(names[i]) + " must be positive");
                sizes_ok = false;
            }
        if (sizes_ok) {
            if (d->n_heads % d->n_kv_heads != 0)
                add(Q3_ERR_UNSUPPORTED_ARCH, "GQA: n_heads (" + std::to_string(d->n_heads) +
                                                 ") is not a multiple of n_kv_heads (" +
                                                 std::to_string(d->n_kv_heads) + ")");
            if (d->hidden % 32 != 0) add(Q3_ERR_UNSUPPORTED_ARCH, "tile alignment: hidden % 32 != 0");
            if (d->intermediate % 32 != 0) add(Q3_ERR_UNSUPPORTED_ARCH, "tile alignment: intermediate % 32 != 0");
            if ((d->n_heads * d->head_dim) % 32 != 0)
                add(Q3_ERR_UNSUPPORTED_ARCH, "tile alignment: n_heads*head_dim % 32 != 0");
            if (d->head_dim != 64 && d->head_dim != 128)
                add(Q3_ERR_UNSUPPORTED_ARCH, "head_dim must be 64 or 128 for these kernels");
            if (d->n_heads % d->n_kv_heads == 0) {
                int gq = d->n_heads / d->n_kv_heads;
                if (gq != 1 && gq != 2 && gq != 4 && gq != 8)
                    add(Q3_ERR_UNSUPPORTED_ARCH, "n_heads/n_kv_heads must be 1, 2, 4 or 8 for these kernels");
            }
            if (d->hidden > 16384 || d->intermediate > 65536)
                add(Q3_ERR_UNSUPPORTED_ARCH, "hidden above 16384 or intermediate above 65536");
        }
        if (d->tie_word_embeddings != 1) add(Q3_ERR_UNSUPPORTED_ARCH, "embeddings: tie_word_embeddings must be true");
        if (d->attention_bias != 0) add(Q3_ERR_UNSUPPORTED_ARCH, "bias: attention bias is not supported");
        if (!(d->rope_theta > 0.f)) add(Q3_ERR_INVALID_ARGUMENTS, "rope_theta must be positive");
        if (!(d->rms_eps >= 0.f)) add(Q3_ERR_INVALID_ARGUMENTS, "rms_eps must be >= 0");
        if (d->max_batch < 1 || d->max_batch > kMaxBatch)
            add(Q3_ERR_INVALID_ARGUMENTS, "max_batch must be in [1, " + std::to_string(kMaxBatch) + "]");
        if (d->max_ctx < 0 || d->max_ctx > kCtxCeiling)
            add(Q3_ERR_CONTEXT, "max_ctx must be in [0, " + std::to_string(kCtxCeiling) + "]");
    }
    if (msg && msg_cap) {
        snprintf(msg, msg_cap, "%s", m.c_str());
    }
    return code;
}

// ------------------------------------------------------------------ weights

// [rows][K] int8 (row-major) + scales -> tile blobs (header of 16 scales,
// then fragment-order bytes q + 128).
static void pack_fragments(const int8_t* w, const float* scale, int rows, int K, uint8_t* out) {
    const int tiles = rows / 16, pairs = K / 32;
    auto work = [&](int t0, int t1) {
        for (int tile = t0; tile < t1; ++tile) {
            uint8_t* hdr = out + (size_t)tile * tile_blob_bytes(K);
            memset(hdr, 0, kTileHeader);
            memcpy(hdr, scale + (size_t)tile * 16, 16 * sizeof(float));
            for (int p = 0; p < pairs; ++p)
                for (int lane = 0; lane < 32; ++lane) {
                    const int g = lane >> 2, t = lane & 3;
                    uint8_t* dst = hdr + kTileHeader + (size_t)p * 512 + lane * 16;
                    for (int ks = 0; ks < 2; ++ks) {
                        const int k0 = p * 32 + ks * 16 + 2 * t;
                        const int8_t* r0 = w + (size_t)(tile * 16 + g) * K;
                        const int8_t* r8 = w + (size_t)(tile * 16 + g + 8) * K;
                        const int8_t v[8] = {r0[k0], r0[k0 + 1], r8[k0], r8[k0 + 1],
                                             r0[k0 + 8], r0[k0 + 9], r8[k0 + 8], r8[k0 + 9]};
                        for (int j = 0; j < 8; ++j) dst[ks * 8 + j] = (uint8_t)((int)v[j] + 128);
                    }
                }
        }
    };
    unsigned nt = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
    if (tiles < 64) nt = 1;
    std::vector<std::thread> th;
    for (unsigned i = 0; i < nt; ++i) {
        int t0 = (int)((long long)tiles * i / nt), t1 = (int)((long long)tiles * (i + 1) / nt);
        th.emplace_back(work, t0, t1);
    }
    for (auto& x : th) x.join();
}

// Upload one (possibly fused) matrix given as host row blocks.
int upload_matrix(q3i8_ctx* c, const std::vector<const int8_t*>& row_src, const std::vector<float>& scales, int K,
                  int pad_rows, DevMat* m, bool keep_raw) {
    const int rows = (int)row_src.size();
    const int prow = ((rows + pad_rows - 1) / pad_rows) * pad_rows;
    std::vector<int8_t> raw((size_t)prow * K, 0);
    for (int r = 0; r < rows; ++r) memcpy(&raw[(size_t)r * K], row_src[r], K);
    std::vector<float> sc(prow, 0.f);
    std::copy(scales.begin(), scales.end(), sc.begin());
    std::vector<uint8_t> frag((size_t)(prow / 16) * tile_blob_bytes(K));
    pack_fragments(raw.data(), sc.data(), prow, K, frag.data());
    m->rows = prow;
    m->valid_rows = rows;
    m->cols = K;
    if (keep_raw) {
        CK(c, cudaMalloc(&m->raw, (size_t)prow * K));
        CK(c, cudaMemcpy(m->raw, raw.data(), raw.size(), cudaMemcpyHostToDevice));
    }
    CK(c, cudaMalloc(&m->frag, frag.size()));
    CK(c, cudaMalloc(&m->scale, (size_t)prow * sizeof(float)));
    CK(c, cudaMemcpy(m->frag, frag.data(), frag.size(), cudaMemcpyHostToDevice));
    CK(c, cudaMemcpy(m->scale, sc.data(), sc.size() * sizeof(float), cudaMemcpyHostToDevice));
    c->weight_bytes_dev += (keep_raw ? 2 : 1) * (size_t)prow * K + (size_t)prow * 4;
    return Q3_OK;
}

static int upload_vec(q3i8_ctx* c, const float* h, int n, float** d) {
    CK(c, cudaMalloc(d, (size_t)n * sizeof(float)));
    CK(c, cudaMemcpy(*d, h, (size_t)n * sizeof(float), cudaMemcpyHostToDevice));
    return Q3_OK;
}

static void free_mat(DevMat& m) {
    cudaFree(m.raw);
    cudaFree(m.frag);
    cudaFree(m.scale);
    m = DevMat{};
}

// ------------------------------------------------------------------ buffers

int ensure_capacity(q3i8_ctx* c, int need_ctx) {
    if (need_ctx > kCtxCeiling)
        return fail(c, Q3_ERR_CONTEXT, "context of %d positions exceeds the %d ceiling", need_ctx, kCtxCeiling);
    int want = std::max(c->cap_request, need_ctx);
    want = (want + kChunkPos - 1) / kChunkPos * kChunkPos;
    if (c->kc && want <= c->cap) return Q3_OK;
    drop_graphs(c);
    cudaFree(c->kc);
    cudaFree(c->vc);
    cudaFree(c->rope);
    c->kc = c->vc = nullptr;
    c->rope = nullptr;
    const q3i8_dims& d = c->d;
    const size_t per = (size_t)d.n_layers * c->bmax * d.n_kv_heads * want * d.head_dim;
    CK(c, cudaMalloc(&c->kc, per * 2));
    CK(c, cudaMalloc(&c->vc, per * 2));
    CK(c, cudaMemsetAsync(c->kc, 0, per * 2, c->stream));
    CK(c, cudaMemsetAsync(c->vc, 0, per * 2, c->stream));
    // RoPE table: frequency, angle, cos and sin in double, rounded to fp32
    const int half = d.head_dim / 2;
    std::vector<float2> tab((size_t)want * half);
    for (int i = 0; i < half; ++i) {
        const double freq = pow((double)d.rope_theta, -2.0 * (double)i / (double)d.head_dim);
        for (int p = 0; p < want; ++p) {
            const double ang = (double)p * freq;
            tab[(size_t)p * half + i] = make_float2((float)cos(ang), (float)sin(ang));
        }
    }
    CK(c, cudaMalloc(&c->rope, tab.size() * sizeof(float2)));
    CK(c, cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice));
    c->cap = want;
    return Q3_OK;
}

static int ensure_out(q3i8_ctx* c, int out_cap) {
    if (c->out_ids && out_cap <= c->out_cap) return Q3_OK;
    drop_graphs(c);
    cudaFree(c->out_ids);
    c->out_ids = nullptr;
    int cap = std::max(out_cap, 256);
    CK(c, cudaMalloc(&c->out_ids, (size_t)c->bmax * cap * sizeof(int32_t)));
    c->out_cap = cap;
    return Q3_OK;
}

static int ensure_prefill(q3i8_ctx* c, int M) {
    if (M <= c->pf_rows) return Q3_OK;
    const q3i8_dims& d = c->d;
    const int H = d.hidden, I = d.intermediate, Dq = d.n_heads * d.head_dim, Dkv = d.n_kv_heads * d.head_dim;
    for (float** p : {&c->pf_x, &c->pf_qkv, &c->pf_q, &c->pf_part}) cudaFree(*p), *p = nullptr;
    for (__half** p : {&c->pf_xh, &c->pf_oh, &c->pf_ah}) cudaFree(*p), *p = nullptr;
    cudaFree(c->pf_ids);
    cudaFree(c->pf_seq);
    cudaFree(c->pf_pos);
    c->pf_rows = 0;
    const size_t m = (size_t)M;
    CK(c, cudaMalloc(&c->pf_x, m * H * 4));
    CK(c, cudaMalloc(&c->pf_qkv, m * (Dq + 2 * Dkv) * 4));
    CK(c, cudaMalloc(&c->pf_q, m * Dq * 4));
    CK(c, cudaMalloc(&c->pf_xh, 2 * m * H * 2));
    CK(c, cudaMalloc(&c->pf_oh, 2 * m * Dq * 2));
    CK(c, cudaMalloc(&c->pf_ah, 2 * m * I * 2));
    cudaFree(c->pf_blocks);
    c->pf_blocks_cap = M / 32 + kMaxBatch + 1;
    CK(c, cudaMalloc(&c->pf_blocks, (size_t)c->pf_blocks_cap * sizeof(int4)));
    CK(c, cudaMalloc(&c->pf_part, attn_part_bytes(M, d.n_heads, d.head_dim, 1)));
    CK(c, cudaMalloc(&c->pf_ids, m * 4));
    CK(c, cudaMalloc(&c->pf_seq, m * 4));
    CK(c, cudaMalloc(&c->pf_pos, m * 4));
    c->pf_rows = M;
    return Q3_OK;
}

void drop_graphs(q3i8_ctx* c) {
    for (auto& kv : c->graphs) cudaGraphExecDestroy(kv.second);
    c->graphs.clear();
}

// ------------------------------------------------------------------ init / destroy

extern "C" int q3i8_init(const q3i8_dims* dims, const q3i8_mat* embed, const q3i8_layer* layers,
                         const float* final_norm, void* cuda_stream, q3i8_ctx** out) {
    if (out) *out = nullptr;
    char msg[1024];
    int rc = q3i8_validate_dims(dims, msg, sizeof msg);
    if (rc != Q3_OK) return fail(nullptr, rc, "%s", msg);
    if (!embed || !embed->w || !embed->scale || !layers || !final_norm || !out)
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "init: a required pointer is NULL");
    for (int l = 0; l < dims->n_layers; ++l) {
        const q3i8_layer& L = layers[l];
        const q3i8_mat* ms[] = {&L.q, &L.k, &L.v, &L.o, &L.gate, &L.up, &L.down};
        for (auto* m : ms)
            if (!m->w || !m->scale) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "init: layer %d has a NULL matrix", l);
        if (!L.attn_norm || !L.ffn_norm || !L.q_norm || !L.k_norm)
            return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "init: layer %d has a NULL norm gain", l);
    }
    int dev = 0, ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
        cudaGetLastError();
        return fail(nullptr, Q3_ERR_NO_DEVICE, "no CUDA device");
    }
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(nullptr, Q3_ERR_NO_DEVICE, "cudaGetDevice failed");
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return fail(nullptr, Q3_ERR_NO_DEVICE, "no device properties");
    if (!(prop.major == 10 && prop.minor == 3))
        return fail(nullptr, Q3_ERR_NO_DEVICE, "device %s is sm_%d%d; this library is built for sm_103a", prop.name,
                    prop.major, prop.minor);

    q3i8_ctx* c = new q3i8_ctx();
    c->d = *dims;
    c->dev = dev;
    c->num_sms = prop.multiProcessorCount;
    c->bmax = dims->max_batch;
    c->cap_request = dims->max_ctx > 0 ? dims->max_ctx : 512;
    if (cuda_stream) {
        c->stream = (cudaStream_t)cuda_stream;
    } else {
        if (cudaStreamCreateWithFlags(&c->stream, cudaStreamNonBlocking) != cudaSuccess) {
            delete c;
            return fail(nullptr, Q3_ERR_CUDA, "cudaStreamCreate failed");
        }
        c->own_stream = true;
    }
    rc = init_weights(c, embed, layers, final_norm);
    if (rc == Q3_OK) rc = init_state(c);
    if (rc == Q3_OK) rc = ensure_capacity(c, c->cap_request);
    if (rc == Q3_OK) rc = ensure_out(c, 256);
    if (rc == Q3_OK) rc = persistent_setup(c);
    if (rc == Q3_OK) rc = step_setup(c);
    if (rc == Q3_OK && cudaStreamSynchronize(c->stream) != cudaSuccess) rc = fail(c, Q3_ERR_CUDA, "init sync failed");
    if (rc != Q3_OK) {
        g_tls_error = c->err;
        q3i8_destroy(c);
        return rc;
    }
    *out = c;
    return Q3_OK;
}

int init_weights(q3i8_ctx* c, const q3i8_mat* embed, const q3i8_layer* layers, const float* final_norm) {
    const q3i8_dims& d = c->d;
    const int H = d.hidden, I = d.intermediate, hd = d.head_dim;
    const int Dq = d.n_heads * hd, Dkv = d.n_kv_heads * hd;
    {
        std::vector<const int8_t*> rows(d.vocab);
        for (int r = 0; r < d.vocab; ++r) rows[r] = embed->w + (size_t)r * H;
        std::vector<float> sc(embed->scale, embed->scale + d.vocab);
        int rc = upload_matrix(c, rows, sc, H, 16, &c->embed, true);
        if (rc) return rc;
    }
    int rc = upload_vec(c, final_norm, H, &c->final_norm);
    if (rc) return rc;
    c->layers.resize(d.n_layers);
    for (int l = 0; l < d.n_layers; ++l) {
        const q3i8_layer& L = layers[l];
        DevLayer& D = c->layers[l];
        std::vector<const int8_t*> rows;
        std::vector<float> sc;
        // fused QKV: rows of Wq, then Wk, then Wv
        for (int r = 0; r < Dq; ++r) rows.push_back(L.q.w + (size_t)r * H), sc.push_back(L.q.scale[r]);
        for (int r = 0; r < Dkv; ++r) rows.push_back(L.k.w + (size_t)r * H), sc.push_back(L.k.scale[r]);
        for (int r = 0; r < Dkv; ++r) rows.push_back(L.v.w + (size_t)r * H), sc.push_back(L.v.scale[r]);
        if ((rc = upload_matrix(c, rows, sc, H, 16, &D.qkv, true))) return rc;
        rows.clear(), sc.clear();
        for (int r = 0; r < H; ++r) rows.push_back(L.o.w + (size_t)r * Dq), sc.push_back(L.o.scale[r]);
        if ((rc = upload_matrix(c, rows, sc, Dq, 16, &D.o, true))) return rc;
        rows.clear(), sc.clear();
        // fused gate/up: blocks of 16 rows = 8 gate units then the same 8 up units
        for (int j = 0; j < I / 8; ++j) {
            for (int r = 0; r < 8; ++r) rows.push_back(L.gate.w + (size_t)(8 * j + r) * H), sc.push_back(L.gate.scale[8 * j + r]);
            for (int r = 0; r < 8; ++r) rows.push_back(L.up.w + (size_t)(8 * j + r) * H), sc.push_back(L.up.scale[8 * j + r]);
        }
        if ((rc = upload_matrix(c, rows, sc, H, 16, &D.gu, true))) return rc;
        rows.clear(), sc.clear();
        for (int r = 0; r < H; ++r) rows.push_back(L.down.w + (size_t)r * I), sc.push_back(L.down.scale[r]);
        if ((rc = upload_matrix(c, rows, sc, I, 16, &D.down, true))) return rc;
        if ((rc = upload_vec(c, L.attn_norm, H, &D.attn_norm))) return rc;
        if ((rc = upload_vec(c, L.ffn_norm, H, &D.ffn_norm))) return rc;
        if ((rc = upload_vec(c, L.q_norm, hd, &D.q_norm))) return rc;
        if ((rc = upload_vec(c, L.k_norm, hd, &D.k_norm))) return rc;
    }
    return Q3_OK;
}

int init_state(q3i8_ctx* c) {
    const q3i8_dims& d = c->d;
    const int H = d.hidden, I = d.intermediate, Dq = d.n_heads * d.head_dim, Dkv = d.n_kv_heads * d.head_dim;
    const int B = c->bmax;
    CK(c, cudaMalloc(&c->tokens, B * 4));
    CK(c, cudaMalloc(&c->pos, B * 4));
    CK(c, cudaMalloc(&c->seq_ids, B * 4));
    CK(c, cudaMalloc(&c->step, 4));
    CK(c, cudaMalloc(&c->keys, B * 8));
    CK(c, cudaMalloc(&c->counter, 4));
    CK(c, cudaMalloc(&c->kpart, (size_t)(H / 16) * kResidSplit * 8 * 64 * sizeof(float)));
    CK(c, cudaMalloc(&c->tile_cnt, (size_t)(H / 16) * sizeof(unsigned int)));
    CK(c, cudaMalloc(&c->ss_fold, (size_t)2 * B * sizeof(long long)));
    CK(c, cudaMemset(c->tile_cnt, 0, (size_t)(H / 16) * sizeof(unsigned int)));
    c->attn_resident = attention_decode_blocks_per_sm(d.head_dim, d.n_heads / d.n_kv_heads) * c->num_sms;
    CK(c, cudaMalloc(&c->status, 4));
    CK(c, cudaMalloc(&c->x, (size_t)B * H * 4));
    CK(c, cudaMalloc(&c->qkv, (size_t)B * (Dq + 2 * Dkv) * 4));
    c->dec_splits_max = 64;
    CK(c, cudaMalloc(&c->part, attn_part_bytes(B, d.n_heads, d.head_dim, c->dec_splits_max)));
    const int K = std::max(std::max(H, I), Dq);
    // activation planes of the chained step: fragment order reserves all 8
    // column tiles (32 sequences) of every k-pair, whatever max_batch is
    const int pcols = 64;
    CK(c, cudaMalloc(&c->xh, (size_t)pcols * K * 2));
    CK(c, cudaMalloc(&c->oh, (size_t)pcols * Dq * 2));
    CK(c, cudaMalloc(&c->ah, (size_t)pcols * I * 2));
    CK(c, cudaMalloc(&c->logits, (size_t)B * d.vocab * 4));
    CK(c, cudaMemsetAsync(c->xh, 0, (size_t)pcols * K * 2, c->stream));
    CK(c, cudaMemsetAsync(c->oh, 0, (size_t)pcols * Dq * 2, c->stream));
    CK(c, cudaMemsetAsync(c->ah, 0, (size_t)pcols * I * 2, c->stream));
    CK(c, cudaMemsetAsync(c->keys, 0, B * 8, c->stream));
    CK(c, cudaMemsetAsync(c->counter, 0, 4, c->stream));
    CK(c, cudaMemsetAsync(c->status, 0, 4, c->stream));
    CK(c, cudaMemsetAsync(c->step, 0, 4, c->stream));
    std::vector<int32_t> ids(B);
    for (int b = 0; b < B; ++b) ids[b] = b;
    CK(c, cudaMemcpy(c->seq_ids, ids.data(), B * 4, cudaMemcpyHostToDevice));
    return Q3_OK;
}

extern "C" void q3i8_destroy(q3i8_ctx* c) {
    if (!c) return;
    cudaStreamSynchronize(c->stream);
    drop_graphs(c);
    free_mat(c->embed);
    for (auto& L : c->layers) {
        free_mat(L.qkv), free_mat(L.o), free_mat(L.gu), free_mat(L.down);
        cudaFree(L.attn_norm), cudaFree(L.ffn_norm), cudaFree(L.q_norm), cudaFree(L.k_norm);
    }
    void* ptrs[] = {c->final_norm, c->kc, c->vc, c->rope, c->tokens, c->pos, c->seq_ids, c->step, c->keys,
                    c->counter, c->kpart, c->tile_cnt, c->ss_fold, c->status, c->x, c->qkv, c->part, c->xh, c->oh, c->ah, c->logits,
                    c->out_ids, c->pf_x, c->pf_qkv, c->pf_q, c->pf_xh, c->pf_oh, c->pf_ah, c->pf_blocks,
                    c->pf_part, c->pf_ids, c->pf_seq, c->pf_pos, c->pf_last, c->d_mats, c->d_gains,
                    c->p_epoch, c->p_keys, c->p_exit, c->p_attn_cnt, c->p_abort, c->p_diag, c->p_ll, c->p_part, c->p_trace,
                    c->xa, c->xf, c->s_params, c->s_counts, c->s_band_key, c->s_band_tok, c->pf_work};
    for (void* p : ptrs) cudaFree(p);
    if (c->ev0) cudaEventDestroy(c->ev0);
    if (c->ev1) cudaEventDestroy(c->ev1);
    if (c->ev2) cudaEventDestroy(c->ev2);
    if (c->own_stream) cudaStreamDestroy(c->stream);
    delete c;
}

// ------------------------------------------------------------------ the decode step

// CTAs per kv head of the decode attention: as many as fill one wave of
// resident attention CTAs, at least one per row, and no more than the rows
// can use (one per 64-position chunk of the capacity, at most
// dec_splits_max per row).  The kernel shares them between the rows by their
// lengths (long rows take several splits, short ones one), so no CTA's split
// is much longer than the others.
int decode_splits(const q3i8_ctx* c, int B) {
    const int per_head = c->attn_resident > 0 ? c->attn_resident / c->d.n_kv_heads : 8 * c->num_sms / c->d.n_kv_heads;
    const int per_row = std::max(1, std::min(c->dec_splits_max, c->cap / kChunkPos));
    return std::max(B, std::min(per_head, B * per_row));
}

// Enqueue one decode step for B sequences: tokens[b] at positions pos[b].
int enqueue_step(q3i8_ctx* c, int B, bool want_logits) {
    const q3i8_dims& d = c->d;
    const int H = d.hidden, I = d.intermediate, hd = d.head_dim, nh = d.n_heads, nkv = d.n_kv_heads;
    const int Dq = nh * hd;
    const size_t layer_kv = (size_t)c->bmax * nkv * c->cap * hd;
    cudaStream_t st = c->stream;
    const int splits = decode_splits(c, B);
    // the residual projections have only hidden/16 tiles: their K is split
    // over kResidSplit CTAs per tile, and the tile's last CTA sums the parts
    // in order, so a step gives the same bits on every run (atomic adds
    // measured about 7 % faster at B = 32, 1.80 vs 1.94 ms per step, but
    // their order, and so their rounding, changes from run to run)
    const int ks_resid = kResidSplit;
    float* kpart = c->kpart;

    // RMSNorm folded (except layer 0's): the residual projections write the
    // next norm's operand planes and per-sequence sums of squares (ss_a after
    // down, ss_b after O); the consumer projections scale by 1 / rms.  Each
    // accumulator is zeroed by a launch between its reader and its next
    // writer: QKV clears ss_b, gate/up clears ss_a.
    long long* ss_a = c->ss_fold;
    long long* ss_b = c->ss_fold + c->bmax;
    launch_embed(c->tokens, B, c->embed.raw, c->embed.scale, H, d.vocab, c->x, c->status, st);
    launch_rmsnorm(c->x, nullptr, B, H, c->layers[0].attn_norm, d.rms_eps, nullptr, c->xh, st, 1);
    for (int l = 0; l < d.n_layers; ++l) {
        const DevLayer& L = c->layers[l];
        GemvArgs a{};
        a.B = B;
        a.w = L.qkv.frag, a.scale = L.qkv.scale, a.rows = L.qkv.rows, a.K = H, a.xh = c->xh, a.xfrag = 1;
        a.y = c->qkv, a.ldy = L.qkv.rows;
        a.ss_in = l > 0 ? ss_a : nullptr, a.ss_clear = ss_b, a.norm_H = H, a.eps = d.rms_eps;
        a.status = c->status;
        // the attention launched next may then read the positions and the
        // cached K/V before its own wait
        a.late_dependents = 1;
        launch_gemv(a, kStore, gemv_grid(a.rows, kStore, c->num_sms), st);
        if (launch_attention_decode(c->qkv, L.q_norm, L.k_norm, d.rms_eps, c->rope, c->kc + l * layer_kv,
                                    c->vc + l * layer_kv, c->seq_ids, c->pos, B, nh, nkv, hd, c->cap, splits,
                                    c->dec_splits_max, c->part, c->oh, Dq, c->status, st, 1))
            return fail(c, Q3_ERR_CUDA, "decode attention could not be launched");
        a = GemvArgs{};
        a.B = B;
        a.w = L.o.frag, a.scale = L.o.scale, a.rows = L.o.rows, a.K = Dq, a.xh = c->oh, a.xfrag = 1;
        a.y = c->x, a.ldy = H, a.ksplit = ks_resid, a.kpart = kpart, a.tile_cnt = c->tile_cnt;
        a.norm_g = L.ffn_norm, a.norm_xh = c->xh, a.ss_out = ss_b, a.norm_H = H;
        a.status = c->status;
        launch_gemv(a, kResid, gemv_grid(a.rows, kResid, c->num_sms) * ks_resid, st);
        a = GemvArgs{};
        a.B = B;
        a.w = L.gu.frag, a.scale = L.gu.scale, a.rows = L.gu.rows, a.K = H, a.xh = c->xh, a.xfrag = 1;
        a.yh = c->ah, a.ldyh = I, a.yfrag = 1;
        a.ss_in = ss_b, a.ss_clear = ss_a, a.norm_H = H, a.eps = d.rms_eps;
        a.status = c->status;
        launch_gemv(a, kSiluGate, gemv_grid(a.rows, kSiluGate, c->num_sms), st);
        a = GemvArgs{};
        a.B = B;
        a.w = L.down.frag, a.scale = L.down.scale, a.rows = L.down.rows, a.K = I, a.xh = c->ah, a.xfrag = 1;
        a.y = c->x, a.ldy = H, a.ksplit = ks_resid, a.kpart = kpart, a.tile_cnt = c->tile_cnt;
        a.norm_g = (l + 1 < d.n_layers) ? c->layers[l + 1].attn_norm : c->final_norm;
        a.norm_xh = c->xh, a.ss_out = ss_a, a.norm_H = H;
        a.status = c->status;
        launch_gemv(a, kResid, gemv_grid(a.rows, kResid, c->num_sms) * ks_resid, st);
    }
    enqueue_lm_head(c, B, true, want_logits ? c->logits : nullptr, ss_a);
    return Q3_OK;
}

void enqueue_lm_head(q3i8_ctx* c, int B, bool advance_pos, float* logits, const long long* ss_in) {
    GemvArgs a{};
    a.B = B;
    a.w = c->embed.frag, a.scale = c->embed.scale, a.rows = c->embed.rows, a.K = c->d.hidden, a.xh = c->xh;
    a.xfrag = 1;  // the final RMSNorm (or the last down projection) writes fragment-ordered planes
    a.ss_in = ss_in, a.norm_H = c->d.hidden, a.eps = c->d.rms_eps;
    a.keys = c->keys, a.counter = c->counter, a.tokens = c->tokens, a.out_ids = c->out_ids, a.step = c->step;
    a.out_cap = c->out_cap, a.pos = c->pos, a.advance_pos = advance_pos ? 1 : 0;
    a.valid_rows = c->embed.valid_rows, a.logits = logits;
    launch_gemv(a, kArgmax, gemv_grid(a.rows, kArgmax, c->num_sms), c->stream);
}

// ------------------------------------------------------------------ small-batch step (step.cu)

static StepShape step_shape(const q3i8_ctx* c) {
    const q3i8_dims& d = c->d;
    return StepShape{d.hidden, d.intermediate, d.n_heads, d.n_kv_heads, d.head_dim, c->embed.rows};
}

// Chooses the launch geometry of the small-batch step and allocates its
// fixed-point residual accumulators.  Q3I8_DECODE_PATH=chained keeps every
// batch on the chained kernels.
int step_setup(q3i8_ctx* c) {
    const char* env = getenv("Q3I8_DECODE_PATH");
    if (env && strcmp(env, "chained") == 0) return Q3_OK;
    int optin = 0;
    CK(c, cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->dev));
    StepPlan p;
    if (!step_plan(step_shape(c), c->num_sms, optin, &p)) return Q3_OK;
    if (!step_prepare_device()) return fail(c, Q3_ERR_CUDA, "decode step kernels: shared-memory opt-in refused");
    if (attn_block_max_clusters(c->d.hidden, c->d.head_dim, p.kv_stages) < 1 ||
        ffn_block_max_blocks(c->d.hidden) < 1)
        return Q3_OK;
    const size_t n = 2 * (size_t)c->bmax * c->d.hidden;  // two buffers each
    CK(c, cudaMalloc(&c->xa, n * sizeof(long long)));
    CK(c, cudaMalloc(&c->xf, n * sizeof(long long)));
    CK(c, cudaMemsetAsync(c->xa, 0, n * sizeof(long long), c->stream));
    CK(c, cudaMemsetAsync(c->xf, 0, n * sizeof(long long), c->stream));
    c->splan = p;
    c->use_step = true;
    // The small-batch kernels are built for up to kStepMaxBatch rows, but from
    // 3 rows on the chained kernels are faster (0.6B shape, prompts of 32-53
    // tokens, 64 new: 460 / 543 / 641 / 735 us per step at B = 1..4 here
    // against 616 / 611 / 615 / 621 us chained).
    c->step_max_batch = 2;
    c->step_max_ctx = 2048;
    if (const char* mc = getenv("Q3I8_STEP_MAX_CTX")) c->step_max_ctx = std::max(0, atoi(mc));
    if (const char* mb = getenv("Q3I8_STEP_MAX_BATCH")) c->step_max_batch = std::max(0, std::min(kStepMaxBatch, atoi(mb)));
    return Q3_OK;
}

// Clears the residual accumulators after a step that did not finish.
static void step_reset(q3i8_ctx* c) {
    if (!c->use_step) return;
    const size_t n = 2 * (size_t)c->bmax * c->d.hidden * sizeof(long long);
    cudaMemsetAsync(c->xa, 0, n, c->stream);
    cudaMemsetAsync(c->xf, 0, n, c->stream);
}

// One decode step for B <= kStepMaxBatch sequences: per layer the attention
// block and the FFN block, then the lm_head.  Layer l accumulates the
// attention block's output in xa[l % 2] and the FFN block's in xf[l % 2];
// a buffer is cleared by a kernel that runs after its last reader and
// before its next writer: the attention block of layer l clears xf[l % 2]
// and xa[(l + 1) % 2], the lm_head clears xa[0] for the next step.
int enqueue_step_fused(q3i8_ctx* c, int B, bool want_logits) {
    const q3i8_dims& d = c->d;
    const int H = d.hidden, I = d.intermediate, hd = d.head_dim, nl = d.n_layers;
    const size_t layer_kv = (size_t)c->bmax * d.n_kv_heads * c->cap * hd;
    const size_t nbuf = (size_t)c->bmax * H;
    const StepPlan& p = c->splan;
    cudaStream_t st = c->stream;
    for (int l = 0; l < nl; ++l) {
        const DevLayer& L = c->layers[l];
        long long* xa = c->xa + (l % 2) * nbuf;
        long long* xf = c->xf + (l % 2) * nbuf;
        AttnBlockArgs a{};
        a.B = B, a.H = H, a.nh = d.n_heads, a.nkv = d.n_kv_heads, a.cap = c->cap, a.kv_stages = p.kv_stages;
        a.vocab = d.vocab;
        a.eps = d.rms_eps;
        a.wqkv = L.qkv.frag, a.qkv_scale = L.qkv.scale, a.wo = L.o.frag, a.o_scale = L.o.scale;
        a.attn_norm = L.attn_norm, a.q_norm = L.q_norm, a.k_norm = L.k_norm, a.rope = c->rope;
        a.kc = c->kc + l * layer_kv, a.vc = c->vc + l * layer_kv;
        a.seq_ids = c->seq_ids, a.pos = c->pos, a.pos_early = l > 0 ? 1 : 0;
        a.xin = l > 0 ? c->xf + ((l - 1) % 2) * nbuf : nullptr;
        a.tokens = c->tokens, a.emb = c->embed.raw, a.emb_scale = c->embed.scale;
        a.xa = xa;
        a.clear0 = xf;
        a.clear1 = l + 1 < nl ? c->xa + ((l + 1) % 2) * nbuf : nullptr;
        a.status = c->status;
        cudaError_t e = launch_attn_block(a, hd, st);
        if (e != cudaSuccess) return fail(c, Q3_ERR_CUDA, "attention block launch: %s", cudaGetErrorString(e));
        FfnBlockArgs f{};
        f.B = B, f.H = H, f.I = I, f.eps = d.rms_eps;
        f.wgu = L.gu.frag, f.gu_scale = L.gu.scale, f.wd = L.down.frag, f.d_scale = L.down.scale;
        f.ffn_norm = L.ffn_norm, f.xa = xa, f.xf = xf, f.status = c->status;
        e = launch_ffn_block(f, p.ffn_grid, st);
        if (e != cudaSuccess) return fail(c, Q3_ERR_CUDA, "FFN block launch: %s", cudaGetErrorString(e));
    }
    LmHeadArgs m{};
    m.B = B, m.H = H, m.rows = c->embed.rows, m.valid_rows = c->embed.valid_rows, m.stages = p.lm_stages;
    m.eps = d.rms_eps;
    m.w = c->embed.frag, m.final_norm = c->final_norm, m.xf = c->xf + ((nl - 1) % 2) * nbuf;
    m.clear = c->xa;
    m.keys = c->keys, m.counter = c->counter, m.tokens = c->tokens, m.out_ids = c->out_ids, m.step = c->step;
    m.out_cap = c->out_cap, m.pos = c->pos, m.advance_pos = 1, m.logits = want_logits ? c->logits : nullptr;
    m.status = c->status;
    cudaError_t e = launch_lm_head(m, p.lm_grid, st);
    if (e != cudaSuccess) return fail(c, Q3_ERR_CUDA, "lm_head launch: %s", cudaGetErrorString(e));
    return Q3_OK;
}

// ------------------------------------------------------------------ persistent step

int persistent_setup(q3i8_ctx* c) {
    const char* env = getenv("Q3I8_DECODE_PATH");
    if (env && strcmp(env, "chained") == 0) return Q3_OK;
    if (!persistent_supported(c->d)) return Q3_OK;
    if (c->d.hidden / 16 > 4 * c->num_sms || c->d.hidden > 4096) return Q3_OK;  // resident H-row tiles
    int optin = 0;
    CK(c, cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->dev));
    const q3i8_dims& d = c->d;
    c->p_kmax = std::max(std::max(d.hidden, d.intermediate), d.n_heads * d.head_dim);
    c->p_optin = optin;
    for (int b = 1; b <= c->bmax; ++b)
        if (persistent_slots(optin, b, c->p_kmax) < 4) return Q3_OK;
    const int ns = persistent_slots(optin, 1, c->p_kmax);
    const int L = d.n_layers, H = d.hidden, I = d.intermediate, hd = d.head_dim;
    const int Dq = d.n_heads * hd, Dkv = d.n_kv_heads * hd, B = c->bmax, G = c->num_sms;
    std::vector<const uint8_t*> mats(4 * L);
    std::vector<const float*> gains(4 * L);
    for (int l = 0; l < L; ++l) {
        mats[4 * l + 0] = c->layers[l].qkv.frag;
        mats[4 * l + 1] = c->layers[l].o.frag;
        mats[4 * l + 2] = c->layers[l].gu.frag;
        mats[4 * l + 3] = c->layers[l].down.frag;
        gains[4 * l + 0] = c->layers[l].attn_norm;
        gains[4 * l + 1] = c->layers[l].ffn_norm;
        gains[4 * l + 2] = c->layers[l].q_norm;
        gains[4 * l + 3] = c->layers[l].k_norm;
    }
    CK(c, cudaMalloc(&c->d_mats, mats.size() * sizeof(void*)));
    CK(c, cudaMalloc(&c->d_gains, gains.size() * sizeof(void*)));
    CK(c, cudaMemcpy(c->d_mats, mats.data(), mats.size() * sizeof(void*), cudaMemcpyHostToDevice));
    CK(c, cudaMemcpy(c->d_gains, gains.data(), gains.size() * sizeof(void*), cudaMemcpyHostToDevice));
    CK(c, cudaMalloc(&c->p_epoch, 4));
    CK(c, cudaMalloc(&c->p_keys, B * 8));
    CK(c, cudaMalloc(&c->p_exit, 4));
    CK(c, cudaMalloc(&c->p_attn_cnt, (size_t)L * B * d.n_kv_heads * 4));
    CK(c, cudaMalloc(&c->p_abort, 4));
    CK(c, cudaMalloc(&c->p_diag, 8 * 4));
    const size_t words = (size_t)B * (3 * H + H / 8 + (Dq + 2 * Dkv) + Dq + I);
    c->p_ll_bytes = words * 8;
    CK(c, cudaMalloc(&c->p_ll, c->p_ll_bytes));
    CK(c, cudaMemset(c->p_ll, 0, c->p_ll_bytes));
    CK(c, cudaMalloc(&c->p_part, (size_t)B * d.n_kv_heads * (G + 1) * 2 * (hd + 2) * sizeof(float)));
    c->p_grid = G;
    c->p_ns = ns;
    if (int rc = persistent_reset(c)) return rc;
    const uint32_t one = 1;
    CK(c, cudaMemcpy(c->p_epoch, &one, 4, cudaMemcpyHostToDevice));
    c->use_persistent = true;
    // Measured on GB300 (0.6B shape): the chained kernels with programmatic
    // dependent launch decode faster at every batch (B = 1: 1.01 vs 1.09 ms
    // per step; B = 8: 1.0 vs 2.0 ms), so by default no batch takes the
    // persistent kernel; Q3I8_PERSISTENT_MAX_BATCH selects it up to that B.
    c->p_max_batch = 0;
    if (const char* mb = getenv("Q3I8_PERSISTENT_MAX_BATCH")) c->p_max_batch = std::max(0, atoi(mb));
    return Q3_OK;
}

// Clear the persistent kernel's between-step state (after init or a timeout)
// and move to a fresh epoch so that no flagged word of an interrupted step
// can match.
int persistent_reset(q3i8_ctx* c) {
    const q3i8_dims& d = c->d;
    CK(c, cudaMemset(c->p_keys, 0, c->bmax * 8));
    CK(c, cudaMemset(c->p_exit, 0, 4));
    CK(c, cudaMemset(c->p_attn_cnt, 0, (size_t)d.n_layers * c->bmax * d.n_kv_heads * 4));
    CK(c, cudaMemset(c->p_abort, 0, 4));
    CK(c, cudaMemset(c->p_diag, 0, 8 * 4));
    uint32_t e = 0;
    CK(c, cudaMemcpy(&e, c->p_epoch, 4, cudaMemcpyDeviceToHost));
    e = (e < 1 ? 1 : e) + 2;
    CK(c, cudaMemcpy(c->p_epoch, &e, 4, cudaMemcpyHostToDevice));
    return Q3_OK;
}

cudaError_t enqueue_persistent(q3i8_ctx* c, int B, float* logits, unsigned long long* trace) {
    const q3i8_dims& d = c->d;
    const int H = d.hidden, I = d.intermediate, hd = d.head_dim;
    const int Dq = d.n_heads * hd, Dkv = d.n_kv_heads * hd, bm = c->bmax;
    PParams P{};
    P.B = B, P.bmax = bm, P.H = H, P.I = I, P.L = d.n_layers, P.nh = d.n_heads, P.nkv = d.n_kv_heads, P.hd = hd;
    P.cap = c->cap, P.vocab = d.vocab, P.vpad = c->embed.rows, P.qkv_rows = c->layers[0].qkv.rows;
    P.kmax = c->p_kmax, P.ns = persistent_slots(c->p_optin, B, c->p_kmax);
    P.eps = d.rms_eps;
    P.mats = c->d_mats, P.lm = c->embed.frag, P.emb_raw = c->embed.raw, P.emb_scale = c->embed.scale;
    P.gains = c->d_gains, P.final_norm = c->final_norm, P.rope = c->rope, P.kc = c->kc, P.vc = c->vc;
    P.tokens = c->tokens, P.pos = c->pos, P.step = c->step, P.out_ids = c->out_ids, P.out_cap = c->out_cap;
    P.advance_pos = 1, P.epoch = c->p_epoch, P.keys = c->p_keys, P.exit_cnt = c->p_exit;
    P.attn_cnt = c->p_attn_cnt, P.status = c->status, P.abort_flag = c->p_abort, P.diag = c->p_diag;
    P.logits = logits;
    P.trace = trace;
    LLw* w = reinterpret_cast<LLw*>(c->p_ll);
    P.x = w, w += (size_t)bm * H;
    P.pl_attn = w, w += (size_t)bm * H;
    P.pl_ffn = w, w += (size_t)bm * H;
    P.ss_attn = w, w += (size_t)bm * (H / 16);
    P.ss_ffn = w, w += (size_t)bm * (H / 16);
    P.qkv = w, w += (size_t)bm * (Dq + 2 * Dkv);
    P.pl_o = w, w += (size_t)bm * Dq;
    P.pl_a = w;
    P.part = c->p_part;
    return launch_persistent_step(P, c->p_grid, c->stream);
}

// One decode step on the context's stream: the persistent kernel when the
// shape allows it, else the chained kernels.
static bool persistent_for(const q3i8_ctx* c, int B) { return c->use_persistent && B <= c->p_max_batch; }

// The small-batch step serves up to step_max_batch sequences whose contexts
// stay within step_max_ctx positions; longer contexts attend faster in the
// chained kernels' split-KV attention (measured: 1.20 vs 1.49 ms per step at
// 4097..6144 positions, B = 1, 0.6B shape).
static bool fused_for(const q3i8_ctx* c, int B) {
    return c->use_step && B <= c->step_max_batch && c->call_ctx <= c->step_max_ctx;
}

static int enqueue_sample(q3i8_ctx* c, int B, const int32_t* step_ptr, int step_value);

static int enqueue_decode_step(q3i8_ctx* c, int B, bool want_logits) {
    if (c->sampling) {
        // the step writes the logits, then the chain draws the token (it
        // overwrites the argmax the lm_head left in tokens[] / out_ids)
        c->sampling = false;
        const int rc = enqueue_decode_step(c, B, true);
        c->sampling = true;
        return rc ? rc : enqueue_sample(c, B, c->step, 0);
    }
    if (persistent_for(c, B)) {
        cudaError_t e = enqueue_persistent(c, B, want_logits ? c->logits : nullptr);
        if (e != cudaSuccess) return fail(c, Q3_ERR_CUDA, "persistent step launch: %s", cudaGetErrorString(e));
        return Q3_OK;
    }
    if (fused_for(c, B)) return enqueue_step_fused(c, B, want_logits);
    return enqueue_step(c, B, want_logits);
}

int step_launches(const q3i8_ctx* c, int B) {
    if (persistent_for(c, B)) return 1;
    if (fused_for(c, B)) return 2 * c->d.n_layers + 1;
    return 2 + c->d.n_layers * (decode_splits(c, B) > B ? 6 : 5) + 1;
}
// Kernels of one prefill over M prompt rows: embed; per layer 2 RMSNorms, the
// QK-norm/RoPE/append, attention split + merge and the 4 projections (one
// tensor-core GEMM each, or one GEMV per chunk of kPrefillChunk rows); final
// RMSNorm and lm_head.
int prefill_launches(const q3i8_ctx* c, int M) {
    const q3i8_dims& d = c->d;
    const int chunks = (M + kPrefillChunk - 1) / kPrefillChunk;
    auto per = [&](int N, int K) {
        if (M > kPrefillChunk && tc_gemm_supported(N, K)) return tc_gemm_splits(M, N, K, c->num_sms) > 1 ? 2 : 1;
        return chunks;
    };
    const int H = d.hidden, I = d.intermediate, Dq = d.n_heads * d.head_dim, Dkv = d.n_kv_heads * d.head_dim;
    const int proj = per(Dq + 2 * Dkv, H) + per(H, Dq) + per(2 * I, H) + per(H, I);
    const int attn = attn_prefill_supported(d.n_heads, d.n_kv_heads, d.head_dim) ? 1 : 2;
    return 1 + d.n_layers * (3 + attn + proj) + 2;
}

// Graph of one decode step at batch B (captured on first use).
static int get_graph(q3i8_ctx* c, int B, cudaGraphExec_t* out) {
    // one graph per batch size, step kind and token choice (argmax or sampled)
    const int key = 4 * B + (c->sampling ? 2 : 0) + (fused_for(c, B) ? 1 : 0);
    auto it = c->graphs.find(key);
    if (it != c->graphs.end()) {
        *out = it->second;
        return Q3_OK;
    }
    cudaGraph_t g;
    CK(c, cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal));
    const int rc = enqueue_decode_step(c, B, false);
    cudaError_t e = cudaStreamEndCapture(c->stream, &g);
    if (rc != Q3_OK) {
        if (e == cudaSuccess) cudaGraphDestroy(g);
        return rc;
    }
    if (e != cudaSuccess) return fail(c, Q3_ERR_CUDA, "graph capture failed: %s", cudaGetErrorString(e));
    cudaGraphExec_t ex;
    e = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return fail(c, Q3_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
    c->graphs[key] = ex;
    *out = ex;
    return Q3_OK;
}

// ------------------------------------------------------------------ sampling

// Host check of the sampling settings; *greedy is set for temperature 0.
static int validate_sampling(q3i8_ctx* c, const q3i8_sampling* s, bool* greedy) {
    if (!s) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sampling settings are NULL");
    const double vals[] = {s->temperature, s->top_p, s->min_p, s->repeat_penalty, s->presence_penalty,
                           s->frequency_penalty};
    for (double v : vals)
        if (!std::isfinite(v)) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sampling: a setting is not finite");
    if (s->temperature < 0) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sampling: temperature < 0");
    *greedy = s->temperature == 0.0;
    if (*greedy) return Q3_OK;
    if (s->top_k < 1 || s->top_k > kSampleMaxTopK)
        return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sampling: top_k %d outside [1, %d]", s->top_k, kSampleMaxTopK);
    if (!(s->top_p > 0 && s->top_p <= 1)) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sampling: top_p outside (0, 1]");
    if (!(s->min_p >= 0 && s->min_p <= 1)) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sampling: min_p outside [0, 1]");
    if (!(s->repeat_penalty > 0)) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sampling: repeat_penalty <= 0");
    return Q3_OK;
}

static SampleParams device_params(const q3i8_sampling& s) {
    SampleParams p{};
    p.temperature = s.temperature, p.top_p = s.top_p, p.min_p = s.min_p, p.repeat_penalty = s.repeat_penalty;
    p.presence_penalty = s.presence_penalty, p.frequency_penalty = s.frequency_penalty;
    p.top_k = s.top_k, p.seed = s.seed;
    return p;
}

// Buffers of the sampling chain for max_batch sequences (first use only).
static int ensure_sampling(q3i8_ctx* c) {
    if (c->s_params) return Q3_OK;
    const size_t V = c->d.vocab, E = sample_band_entries(c->d.vocab);
    CK(c, cudaMalloc(&c->s_counts, (size_t)c->bmax * V * 4));
    CK(c, cudaMalloc(&c->s_band_key, (size_t)c->bmax * E * 8));
    CK(c, cudaMalloc(&c->s_band_tok, (size_t)c->bmax * E * 4));
    CK(c, cudaMalloc(&c->s_params, sizeof(SampleParams)));
    return Q3_OK;
}

// The chain over c->logits for B sequences: the draw is for generated token
// *step_ptr - 1 (or step_value when step_ptr is NULL).
static int enqueue_sample(q3i8_ctx* c, int B, const int32_t* step_ptr, int step_value) {
    SampleArgs a{};
    a.logits = c->logits, a.ldz = c->d.vocab, a.V = c->d.vocab, a.counts = c->s_counts, a.params = c->s_params;
    a.step = step_ptr, a.step_value = step_value, a.tokens = c->tokens, a.out_ids = c->out_ids, a.out_cap = c->out_cap;
    a.band_key = c->s_band_key, a.band_tok = c->s_band_tok, a.status = c->status;
    cudaError_t e = launch_sample(a, B, c->stream);
    if (e != cudaSuccess) return fail(c, Q3_ERR_CUDA, "sampling launch: %s", cudaGetErrorString(e));
    return Q3_OK;
}

// ------------------------------------------------------------------ prefill

// Prefill B prompts given back to back in device memory; leaves the first
// generated token of each sequence in tokens[] / out_ids[:, 0] (step = 1)
// and pos[b] = prompt length.
static int restore_seq_ids(q3i8_ctx* c);
// scheduler internals (sched.cu)
int q3_sched_slots(const q3i8_sched* s);
int q3_sched_max_ctx(const q3i8_sched* s);
const int32_t* q3_sched_prompt(const q3i8_sched* s, int request_id, int32_t* len);

// slots: the KV cache sequence of prompt b (NULL: b itself, the plain
// decode's layout); other sequences' cache entries are not touched.
static int run_prefill(q3i8_ctx* c, int B, const int32_t* d_ids, const int32_t* lens, float* d_logits,
                       const int32_t* slots = nullptr) {
    const q3i8_dims& d = c->d;
    const int H = d.hidden, I = d.intermediate, hd = d.head_dim, nh = d.n_heads, nkv = d.n_kv_heads;
    const int Dq = nh * hd, Dkv = nkv * hd;
    int M = 0, maxlen = 0;
    for (int b = 0; b < B; ++b) M += lens[b], maxlen = std::max(maxlen, lens[b]);
    int rc = ensure_prefill(c, M);
    if (rc) return rc;
    if (!slots && (rc = restore_seq_ids(c))) return rc;
    cudaStream_t st = c->stream;
    std::vector<int32_t> seq(M), pos(M), last(B), plen(lens, lens + B);
    for (int b = 0, r = 0; b < B; ++b) {
        for (int t = 0; t < lens[b]; ++t, ++r) seq[r] = slots ? slots[b] : b, pos[r] = t;
        last[b] = r - 1;
    }
    if (!c->pf_last) CK(c, cudaMalloc(&c->pf_last, kMaxBatch * 4));
    CK(c, cudaMemcpyAsync(c->pf_seq, seq.data(), M * 4, cudaMemcpyHostToDevice, st));
    CK(c, cudaMemcpyAsync(c->pf_pos, pos.data(), M * 4, cudaMemcpyHostToDevice, st));
    CK(c, cudaMemcpyAsync(c->pf_last, last.data(), B * 4, cudaMemcpyHostToDevice, st));
    CK(c, cudaMemcpyAsync(c->pos, plen.data(), B * 4, cudaMemcpyHostToDevice, st));
    CK(c, cudaMemsetAsync(c->step, 0, 4, st));
    CK(c, cudaMemsetAsync(c->status, 0, 4, st));
    const size_t layer_kv = (size_t)c->bmax * nkv * c->cap * hd;

    // split-K workspace of the tensor-core projections (short prompts on few output tiles)
    if (M > kPrefillChunk) {
        size_t need = 0;
        const int shapes[4][2] = {{Dq + 2 * Dkv, H}, {H, Dq}, {2 * I, H}, {H, I}};
        for (const auto& sh : shapes) need = std::max(need, tc_gemm_work_bytes(M, sh[0], sh[1], c->num_sms));
        if (need > c->pf_work_bytes) {
            cudaFree(c->pf_work);
            c->pf_work = nullptr, c->pf_work_bytes = 0;
            CK(c, cudaMalloc(&c->pf_work, need));
            c->pf_work_bytes = need;
        }
    }
    // One projection over all prompt rows: the tcgen05 GEMM when there is
    // more than one chunk of rows, else the decode GEMV (one weight sweep per
    // chunk of up to kPrefillChunk rows).
    int tc_rc = 0;
    auto project = [&](const DevMat& W, int K, const __half* xh, int mode, float* y, int ldy, __half* yh, int ldyh) {
        if (M > kPrefillChunk && W.raw && tc_gemm_supported(W.rows, K)) {
            const int rc = launch_tc_gemm(xh, W.raw, W.scale, M, W.rows, K, mode, y, ldy, yh, ldyh, c->status, st,
                                          c->pf_work, c->pf_work_bytes, c->num_sms);
            if (rc == 0) return;
            tc_rc = rc;
        }
        for (int m0 = 0; m0 < M; m0 += kPrefillChunk) {
            GemvArgs a{};
            a.B = std::min(kPrefillChunk, M - m0);
            a.w = W.frag, a.scale = W.scale, a.rows = W.rows, a.K = K;
            a.xh = xh + (size_t)2 * m0 * K;
            if (y) a.y = y + (size_t)m0 * ldy, a.ldy = ldy;
            if (yh) a.yh = yh + (size_t)2 * m0 * ldyh, a.ldyh = ldyh;
            a.status = c->status;
            // the residual projections split K over a cluster of CTAs, as in the decode step
            const int ks = mode == kResid ? kResidSplit : 1;
            a.ksplit = ks;
            launch_gemv(a, mode, gemv_grid(a.rows, mode, c->num_sms) * ks, st);
        }
    };
    // causal attention: the tensor-core kernel over 32-position query blocks
    // where the shape allows, else the split kernel with one split per row
    int nblk = 0;
    const bool tc_attn = attn_prefill_supported(nh, nkv, hd);
    if (tc_attn) {
        std::vector<int4> blk(c->pf_blocks_cap);
        nblk = attn_prefill_blocks(lens, B, blk.data(), c->pf_blocks_cap, slots);
        if (nblk > c->pf_blocks_cap) return fail(c, Q3_ERR_STATE, "prefill: query block table too small");
        CK(c, cudaMemcpyAsync(c->pf_blocks, blk.data(), (size_t)nblk * sizeof(int4), cudaMemcpyHostToDevice, st));
        CK(c, cudaStreamSynchronize(st));  // blk is a host temporary
    }
    launch_embed(d_ids, M, c->embed.raw, c->embed.scale, H, d.vocab, c->pf_x, c->status, st);
    for (int l = 0; l < d.n_layers; ++l) {
        const DevLayer& L = c->layers[l];
        launch_rmsnorm(c->pf_x, nullptr, M, H, L.attn_norm, d.rms_eps, nullptr, c->pf_xh, st);
        project(L.qkv, H, c->pf_xh, kStore, c->pf_qkv, L.qkv.rows, nullptr, 0);
        launch_qk_rope_append(c->pf_qkv, M, nh, nkv, hd, c->pf_seq, c->pf_pos, L.q_norm, L.k_norm, d.rms_eps,
                              c->rope, c->pf_q, c->kc + l * layer_kv, c->vc + l * layer_kv, c->cap, st);
        if (tc_attn) {
            if (launch_attn_prefill(c->pf_q, c->kc + l * layer_kv, c->vc + l * layer_kv, c->pf_blocks, nblk, nh, nkv,
                                    hd, c->cap, c->pf_oh, Dq, st))
                return fail(c, Q3_ERR_CUDA, "prefill attention could not be launched");
        } else {
            launch_attention(c->pf_q, c->kc + l * layer_kv, c->vc + l * layer_kv, c->pf_seq, c->pf_pos, 1, M, nh,
                             nkv, hd, c->cap, 1, c->pf_part, nullptr, c->pf_oh, Dq, c->status, st);
        }
        project(L.o, Dq, c->pf_oh, kResid, c->pf_x, H, nullptr, 0);
        launch_rmsnorm(c->pf_x, nullptr, M, H, L.ffn_norm, d.rms_eps, nullptr, c->pf_xh, st);
        project(L.gu, H, c->pf_xh, kSiluGate, nullptr, 0, c->pf_ah, I);
        project(L.down, I, c->pf_ah, kResid, c->pf_x, H, nullptr, 0);
        (void)Dkv;
    }
    if (tc_rc) return fail(c, Q3_ERR_CUDA, "prefill: tensor-core GEMM could not be set up (%d)", tc_rc);
    launch_rmsnorm(c->pf_x, c->pf_last, B, H, c->final_norm, d.rms_eps, nullptr, c->xh, st, 1);
    enqueue_lm_head(c, B, false, d_logits);
    CK(c, cudaGetLastError());
    c->launches += prefill_launches(c, M);
    c->active_B = B;
    c->seq_len.assign(lens, lens + B);
    (void)maxlen;
    return Q3_OK;
}

static int check_status(q3i8_ctx* c) {
    int32_t st = 0;
    CK(c, cudaMemcpyAsync(&st, c->status, 4, cudaMemcpyDeviceToHost, c->stream));
    CK(c, cudaStreamSynchronize(c->stream));
    if (st != 0) {
        cudaMemsetAsync(c->status, 0, 4, c->stream);
        cudaStreamSynchronize(c->stream);
        int32_t dg[8] = {0};
        if (c->use_persistent) {
            cudaMemcpy(dg, c->p_diag, sizeof dg, cudaMemcpyDeviceToHost);
            persistent_reset(c);
        }
        step_reset(c);
        cudaStreamSynchronize(c->stream);
        if (st == kStatusSampleSelect)
            return fail(c, Q3_ERR_CUDA, "sampling: the top-k selection did not add up (internal error)");
        if (st == kStatusBadToken)
            return fail(c, Q3_ERR_INVALID_ARGUMENTS, "a token id outside [0, %d) reached the device", c->d.vocab);
        return fail(c, Q3_ERR_TIMEOUT,
                    "a bounded device wait gave up (status %d; site %d cta %d warp %d layer %d phase %d aux %d)", st,
                    dg[0], dg[1], dg[2], dg[3], dg[4], dg[5]);
    }
    return Q3_OK;
}

static int validate_prompts(q3i8_ctx* c, int B, const int32_t* lens, int max_new, int* need) {
    if (B < 1 || B > c->bmax) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "B=%d outside [1, max_batch=%d]", B, c->bmax);
    if (!lens) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "prompt_lens is NULL");
    if (max_new < 1) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "max_new_tokens < 1");
    int mx = 0;
    for (int b = 0; b < B; ++b) {
        if (lens[b] < 1) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sequence %d: empty prompt", b);
        mx = std::max(mx, lens[b]);
    }
    const long long n = (long long)mx + max_new;
    if (n > kCtxCeiling)
        return fail(c, Q3_ERR_CONTEXT, "prompt (%d) + new tokens (%d) exceeds the %d-position ceiling", mx, max_new,
                    kCtxCeiling);
    *need = (int)n;
    return Q3_OK;
}

static int ensure_events(q3i8_ctx* c) {
    if (!c->ev0) {
        CK(c, cudaEventCreate(&c->ev0));
        CK(c, cudaEventCreate(&c->ev1));
        CK(c, cudaEventCreate(&c->ev2));
    }
    return Q3_OK;
}

// Prefill, then decode steps until max_new tokens per sequence exist or,
// with eos_id >= 0, until every sequence has produced eos_id: the step graph
// is then replayed in chunks of kEosChunk steps and the chunk's ids are read
// back to see whether all sequences are done.  *steps_run receives the
// number of decode steps run.
constexpr int kEosChunk = 16;

static int decode_core(q3i8_ctx* c, int B, const int32_t* d_ids, const int32_t* lens, int max_new, int need,
                       int32_t eos_id, q3i8_stats* stats, int* steps_run = nullptr) {
    int rc = ensure_events(c);
    if (rc) return rc;
    c->call_ctx = need;
    CK(c, cudaEventRecord(c->ev0, c->stream));
    rc = run_prefill(c, B, d_ids, lens, c->sampling ? c->logits : nullptr);
    if (rc) return rc;
    if (c->sampling) {
        // count the prompt tokens of each sequence, then draw token 0
        int M = 0;
        for (int b = 0; b < B; ++b) M += lens[b];
        CK(c, cudaMemsetAsync(c->s_counts, 0, (size_t)B * c->d.vocab * 4, c->stream));
        CK(c, launch_count_tokens(d_ids, c->pf_seq, M, c->s_counts, c->d.vocab, c->stream));
        if ((rc = enqueue_sample(c, B, c->step, 0))) return rc;
        c->launches += 2;
    }
    CK(c, cudaEventRecord(c->ev1, c->stream));
    int steps = 0;
    if (max_new > 1) {
        cudaGraphExec_t g;
        rc = get_graph(c, B, &g);
        if (rc) return rc;
        if (eos_id < 0) {
            for (int i = 1; i < max_new; ++i) CK(c, cudaGraphLaunch(g, c->stream));
            steps = max_new - 1;
        } else {
            std::vector<char> done(B, 0);
            std::vector<int32_t> ids((size_t)B * kEosChunk);
            int col = 0;  // next out_ids column to inspect (column 0 is the prefill's token)
            while (true) {
                const int ncols = std::min(kEosChunk, steps + 1 - col);
                if (ncols > 0) {
                    CK(c, cudaMemcpy2DAsync(ids.data(), (size_t)ncols * 4, c->out_ids + col, (size_t)c->out_cap * 4,
                                            (size_t)ncols * 4, B, cudaMemcpyDeviceToHost, c->stream));
                    CK(c, cudaStreamSynchronize(c->stream));
                    for (int b = 0; b < B; ++b)
                        for (int j = 0; j < ncols; ++j) done[b] |= ids[(size_t)b * ncols + j] == eos_id;
                    col += ncols;
                }
                if (std::all_of(done.begin(), done.end(), [](char d) { return d != 0; }) || steps >= max_new - 1)
                    break;
                const int n = std::min(kEosChunk, max_new - 1 - steps);
                for (int i = 0; i < n; ++i) CK(c, cudaGraphLaunch(g, c->stream));
                steps += n;
            }
        }
        c->launches += (int64_t)steps * (step_launches(c, B) + (c->sampling ? 1 : 0));
    }
    CK(c, cudaEventRecord(c->ev2, c->stream));
    rc = check_status(c);
    if (rc) return rc;
    if (steps_run) *steps_run = steps;
    for (int b = 0; b < B; ++b) c->seq_len[b] += steps;
    if (stats) {
        float pf = 0, dc = 0;
        CK(c, cudaEventElapsedTime(&pf, c->ev0, c->ev1));
        CK(c, cudaEventElapsedTime(&dc, c->ev1, c->ev2));
        long long ptoks = 0;
        for (int b = 0; b < B; ++b) ptoks += lens[b];
        stats->prefill_ms = pf;
        stats->decode_ms = dc;
        stats->prefill_tokens = ptoks;
        stats->decode_steps = steps;
        stats->prefill_tokens_per_sec = pf > 0 ? ptoks / (pf * 1e-3) : 0;
        stats->decode_tokens_per_sec = (dc > 0 && steps > 0) ? (double)B * steps / (dc * 1e-3) : 0;
        stats->step_us = steps > 0 ? dc * 1e3 / steps : 0;
    }
    return Q3_OK;
}

extern "C" int q3i8_decode_device(q3i8_ctx* c, int32_t B, const int32_t* d_prompt_ids, const int32_t* prompt_lens,
                                  int32_t max_new_tokens, int32_t* d_out_ids, q3i8_stats* stats) {
    if (!c) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "ctx is NULL");
    int need = 0;
    int rc = validate_prompts(c, B, prompt_lens, max_new_tokens, &need);
    if (rc) return rc;
    if (!d_prompt_ids || !d_out_ids) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "device id buffer is NULL");
    if ((rc = ensure_capacity(c, need))) return rc;
    if ((rc = ensure_out(c, max_new_tokens))) return rc;
    if ((rc = decode_core(c, B, d_prompt_ids, prompt_lens, max_new_tokens, need, -1, stats))) return rc;
    CK(c, cudaMemcpy2DAsync(d_out_ids, (size_t)max_new_tokens * 4, c->out_ids, (size_t)c->out_cap * 4,
                            (size_t)max_new_tokens * 4, B, cudaMemcpyDeviceToDevice, c->stream));
    CK(c, cudaStreamSynchronize(c->stream));
    return Q3_OK;
}

// Decode with host buffers (q3i8_decode, q3i8_decode_sample).
static int decode_host(q3i8_ctx* c, int32_t B, const int32_t* const* prompt_ids, const int32_t* prompt_lens,
                       int32_t max_new_tokens, int32_t eos_id, int32_t* out_ids, int32_t* out_counts,
                       q3i8_stats* stats) {
    int need = 0;
    int rc = validate_prompts(c, B, prompt_lens, max_new_tokens, &need);
    if (rc) return rc;
    if (!prompt_ids || !out_ids) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "prompt_ids or out_ids is NULL");
    std::vector<int32_t> all;
    for (int b = 0; b < B; ++b) {
        if (!prompt_ids[b]) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "prompt_ids[%d] is NULL", b);
        for (int t = 0; t < prompt_lens[b]; ++t) {
            const int32_t id = prompt_ids[b][t];
            if (id < 0 || id >= c->d.vocab)
                return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sequence %d position %d: id %d outside [0, %d)", b, t, id,
                            c->d.vocab);
            all.push_back(id);
        }
    }
    if ((rc = ensure_capacity(c, need))) return rc;
    if ((rc = ensure_out(c, max_new_tokens))) return rc;
    if ((rc = ensure_prefill(c, (int)all.size()))) return rc;
    CK(c, cudaMemcpyAsync(c->pf_ids, all.data(), all.size() * 4, cudaMemcpyHostToDevice, c->stream));
    int steps = 0;
    if ((rc = decode_core(c, B, c->pf_ids, prompt_lens, max_new_tokens, need, eos_id, stats, &steps))) return rc;
    const int made = steps + 1;  // ids produced per sequence
    CK(c, cudaMemcpy2DAsync(out_ids, (size_t)max_new_tokens * 4, c->out_ids, (size_t)c->out_cap * 4,
                            (size_t)made * 4, B, cudaMemcpyDeviceToHost, c->stream));
    CK(c, cudaStreamSynchronize(c->stream));
    for (int b = 0; b < B; ++b) {
        int n = made;
        if (eos_id >= 0)
            for (int i = 0; i < made; ++i)
                if (out_ids[(size_t)b * max_new_tokens + i] == eos_id) {
                    n = i + 1;
                    break;
                }
        for (int i = made; i < max_new_tokens; ++i) out_ids[(size_t)b * max_new_tokens + i] = -1;
        if (out_counts) out_counts[b] = n;
    }
    return Q3_OK;
}

extern "C" int q3i8_decode(q3i8_ctx* c, int32_t B, const int32_t* const* prompt_ids, const int32_t* prompt_lens,
                           int32_t max_new_tokens, int32_t eos_id, int32_t* out_ids, int32_t* out_counts,
                           q3i8_stats* stats) {
    if (!c) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "ctx is NULL");
    return decode_host(c, B, prompt_ids, prompt_lens, max_new_tokens, eos_id, out_ids, out_counts, stats);
}

extern "C" int q3i8_decode_sample(q3i8_ctx* c, int32_t B, const int32_t* const* prompt_ids,
                                  const int32_t* prompt_lens, int32_t max_new_tokens, int32_t eos_id,
                                  const q3i8_sampling* sampling, int32_t* out_ids, int32_t* out_counts,
                                  q3i8_stats* stats) {
    if (!c) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "ctx is NULL");
    bool greedy = false;
    int rc = validate_sampling(c, sampling, &greedy);
    if (rc) return rc;
    if (greedy) return decode_host(c, B, prompt_ids, prompt_lens, max_new_tokens, eos_id, out_ids, out_counts, stats);
    if ((rc = ensure_sampling(c))) return rc;
    const SampleParams p = device_params(*sampling);
    CK(c, cudaMemcpyAsync(c->s_params, &p, sizeof p, cudaMemcpyHostToDevice, c->stream));
    CK(c, cudaStreamSynchronize(c->stream));  // p is a host temporary
    c->sampling = true;
    rc = decode_host(c, B, prompt_ids, prompt_lens, max_new_tokens, eos_id, out_ids, out_counts, stats);
    c->sampling = false;
    return rc;
}

extern "C" int q3i8_prefill(q3i8_ctx* c, int32_t B, const int32_t* const* prompt_ids, const int32_t* prompt_lens,
                            float* last_logits) {
    if (!c) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "ctx is NULL");
    int need = 0;
    int rc = validate_prompts(c, B, prompt_lens, 1, &need);
    if (rc) return rc;
    if (!prompt_ids) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "prompt_ids is NULL");
    std::vector<int32_t> all;
    for (int b = 0; b < B; ++b) {
        if (!prompt_ids[b]) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "prompt_ids[%d] is NULL", b);
        for (int t = 0; t < prompt_lens[b]; ++t) {
            const int32_t id = prompt_ids[b][t];
            if (id < 0 || id >= c->d.vocab)
                return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sequence %d position %d: id %d outside [0, %d)", b, t, id,
                            c->d.vocab);
            all.push_back(id);
        }
    }
    if ((rc = ensure_capacity(c, need))) return rc;
    if ((rc = ensure_out(c, 256))) return rc;
    if ((rc = ensure_prefill(c, (int)all.size()))) return rc;
    CK(c, cudaMemcpyAsync(c->pf_ids, all.data(), all.size() * 4, cudaMemcpyHostToDevice, c->stream));
    if ((rc = run_prefill(c, B, c->pf_ids, prompt_lens, last_logits ? c->logits : nullptr))) return rc;
    if (last_logits)
        CK(c, cudaMemcpyAsync(last_logits, c->logits, (size_t)B * c->d.vocab * 4, cudaMemcpyDeviceToHost, c->stream));
    return check_status(c);
}

extern "C" int q3i8_step_logits(q3i8_ctx* c, const int32_t* tokens, float* logits) {
    if (!c) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "ctx is NULL");
    if (c->active_B <= 0) return fail(c, Q3_ERR_STATE, "q3i8_step_logits before q3i8_prefill");
    if (!tokens || !logits) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "tokens or logits is NULL");
    const int B = c->active_B;
    for (int b = 0; b < B; ++b) {
        if (tokens[b] < 0 || tokens[b] >= c->d.vocab)
            return fail(c, Q3_ERR_INVALID_ARGUMENTS, "token %d of sequence %d outside [0, %d)", tokens[b], b,
                        c->d.vocab);
        if (c->seq_len[b] + 1 > c->cap)
            return fail(c, Q3_ERR_STATE, "sequence %d is at the context capacity (%d)", b, c->cap);
    }
    c->call_ctx = 1 + *std::max_element(c->seq_len.begin(), c->seq_len.begin() + B);
    CK(c, cudaMemcpyAsync(c->tokens, tokens, B * 4, cudaMemcpyHostToDevice, c->stream));
    if (int rc0 = enqueue_decode_step(c, B, true)) return rc0;
    c->launches += step_launches(c, B);
    CK(c, cudaGetLastError());
    CK(c, cudaMemcpyAsync(logits, c->logits, (size_t)B * c->d.vocab * 4, cudaMemcpyDeviceToHost, c->stream));
    int rc = check_status(c);
    if (rc) return rc;
    for (int b = 0; b < B; ++b) c->seq_len[b] += 1;
    return Q3_OK;
}

// ------------------------------------------------------------------ continuous batching

// Sequence ids of the decode rows back to 0 .. max_batch - 1 (the plain
// calls' layout) after continuous-batching steps pointed them at slots.
static int restore_seq_ids(q3i8_ctx* c) {
    if (!c->seq_ids_custom) return Q3_OK;
    std::vector<int32_t> ids(c->bmax);
    for (int b = 0; b < c->bmax; ++b) ids[b] = b;
    CK(c, cudaMemcpyAsync(c->seq_ids, ids.data(), c->bmax * 4, cudaMemcpyHostToDevice, c->stream));
    CK(c, cudaStreamSynchronize(c->stream));  // ids is a host temporary
    c->seq_ids_custom = false;
    return Q3_OK;
}

extern "C" int q3i8_cb_reserve(q3i8_ctx* c, int32_t max_ctx) {
    if (!c) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "ctx is NULL");
    if (max_ctx < 1) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "cb_reserve: max_ctx < 1");
    int rc = ensure_capacity(c, max_ctx);
    if (rc) return rc;
    return ensure_out(c, 256);
}

extern "C" int q3i8_cb_prefill(q3i8_ctx* c, int32_t n, const int32_t* slots, const int32_t* const* prompt_ids,
                               const int32_t* prompt_lens, int32_t* first_tokens) {
    if (!c) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "ctx is NULL");
    if (n < 1 || n > c->bmax) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "cb_prefill: n=%d outside [1, %d]", n, c->bmax);
    if (!slots || !prompt_ids || !prompt_lens || !first_tokens)
        return fail(c, Q3_ERR_INVALID_ARGUMENTS, "cb_prefill: NULL argument");
    if (!c->kc) return fail(c, Q3_ERR_STATE, "cb_prefill before q3i8_cb_reserve");
    std::vector<char> used(c->bmax, 0);
    std::vector<int32_t> all;
    for (int b = 0; b < n; ++b) {
        if (slots[b] < 0 || slots[b] >= c->bmax || used[slots[b]])
            return fail(c, Q3_ERR_INVALID_ARGUMENTS, "cb_prefill: slot %d invalid or repeated", slots[b]);
        used[slots[b]] = 1;
        if (!prompt_ids[b] || prompt_lens[b] < 1)
            return fail(c, Q3_ERR_INVALID_ARGUMENTS, "cb_prefill: prompt %d is NULL or empty", b);
        if (prompt_lens[b] > c->cap)
            return fail(c, Q3_ERR_CONTEXT, "cb_prefill: prompt %d (%d) exceeds the reserved %d positions", b,
                        prompt_lens[b], c->cap);
        for (int t = 0; t < prompt_lens[b]; ++t) {
            const int32_t id = prompt_ids[b][t];
            if (id < 0 || id >= c->d.vocab)
                return fail(c, Q3_ERR_INVALID_ARGUMENTS, "cb_prefill: prompt %d position %d: id %d outside [0, %d)",
                            b, t, id, c->d.vocab);
            all.push_back(id);
        }
    }
    int rc = ensure_prefill(c, (int)all.size());
    if (rc) return rc;
    CK(c, cudaMemcpyAsync(c->pf_ids, all.data(), all.size() * 4, cudaMemcpyHostToDevice, c->stream));
    if ((rc = run_prefill(c, n, c->pf_ids, prompt_lens, nullptr, slots))) return rc;
    c->active_B = 0;  // the step-by-step interface has no session after this
    CK(c, cudaMemcpyAsync(first_tokens, c->tokens, n * 4, cudaMemcpyDeviceToHost, c->stream));
    return check_status(c);
}

extern "C" int q3i8_cb_step(q3i8_ctx* c, int32_t n, const int32_t* row_slot, const int32_t* row_pos,
                            const int32_t* row_token, int32_t* next_tokens) {
    if (!c) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "ctx is NULL");
    if (n < 1 || n > c->bmax) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "cb_step: n=%d outside [1, %d]", n, c->bmax);
    if (!row_slot || !row_pos || !row_token || !next_tokens)
        return fail(c, Q3_ERR_INVALID_ARGUMENTS, "cb_step: NULL argument");
    if (!c->kc) return fail(c, Q3_ERR_STATE, "cb_step before q3i8_cb_reserve");
    std::vector<char> used(c->bmax, 0);
    int top = 0;
    for (int r = 0; r < n; ++r) {
        if (row_slot[r] < 0 || row_slot[r] >= c->bmax || used[row_slot[r]])
            return fail(c, Q3_ERR_INVALID_ARGUMENTS, "cb_step: slot %d invalid or repeated", row_slot[r]);
        used[row_slot[r]] = 1;
        if (row_pos[r] < 1 || row_pos[r] >= c->cap)
            return fail(c, Q3_ERR_CONTEXT, "cb_step: row %d position %d outside [1, %d)", r, row_pos[r], c->cap);
        if (row_token[r] < 0 || row_token[r] >= c->d.vocab)
            return fail(c, Q3_ERR_INVALID_ARGUMENTS, "cb_step: row %d token %d outside [0, %d)", r, row_token[r],
                        c->d.vocab);
        top = std::max(top, row_pos[r] + 1);
    }
    int rc = ensure_events(c);
    if (rc) return rc;
    c->call_ctx = top;
    c->seq_ids_custom = true;
    cudaStream_t st = c->stream;
    CK(c, cudaMemcpyAsync(c->tokens, row_token, n * 4, cudaMemcpyHostToDevice, st));
    CK(c, cudaMemcpyAsync(c->pos, row_pos, n * 4, cudaMemcpyHostToDevice, st));
    CK(c, cudaMemcpyAsync(c->seq_ids, row_slot, n * 4, cudaMemcpyHostToDevice, st));
    cudaGraphExec_t g;
    if ((rc = get_graph(c, n, &g))) return rc;
    CK(c, cudaGraphLaunch(g, st));
    c->launches += step_launches(c, n);
    CK(c, cudaMemcpyAsync(next_tokens, c->tokens, n * 4, cudaMemcpyDeviceToHost, st));
    return check_status(c);
}

extern "C" int q3i8_sched_run(q3i8_ctx* c, q3i8_sched* s, q3i8_stats* stats) {
    if (!c) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "ctx is NULL");
    if (!s) return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sched_run: scheduler is NULL");
    if (q3_sched_slots(s) > c->bmax)
        return fail(c, Q3_ERR_INVALID_ARGUMENTS, "sched_run: %d slots exceed max_batch %d", q3_sched_slots(s), c->bmax);
    int rc = q3i8_cb_reserve(c, q3_sched_max_ctx(s));
    if (rc) return rc;
    const int nb = c->bmax;
    std::vector<int32_t> a_req(nb), a_slot(nb), r_req(nb), r_slot(nb), r_pos(nb), r_tok(nb), out(nb), lens(nb);
    std::vector<const int32_t*> ptrs(nb);
    int64_t prefill_tokens = 0, steps = 0, step_rows = 0;
    double prefill_ms = 0, decode_ms = 0;
    auto now_ms = [] { return std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now().time_since_epoch()).count(); };
    while (!q3i8_sched_idle(s)) {
        int32_t na = 0, nr = 0;
        if ((rc = q3i8_sched_plan(s, &na, a_req.data(), a_slot.data(), &nr, r_req.data(), r_slot.data(), r_pos.data(),
                                  r_tok.data())))
            return fail(c, rc, "sched_run: %s", q3i8_last_error(nullptr));
        if (na > 0) {
            for (int i = 0; i < na; ++i) {
                int32_t len = 0;
                ptrs[i] = q3_sched_prompt(s, a_req[i], &len);
                lens[i] = len;
                prefill_tokens += len;
            }
            const double t0 = now_ms();
            if ((rc = q3i8_cb_prefill(c, na, a_slot.data(), ptrs.data(), lens.data(), out.data()))) return rc;
            prefill_ms += now_ms() - t0;
            if ((rc = q3i8_sched_complete_prefill(s, na, a_req.data(), out.data())))
                return fail(c, rc, "sched_run: %s", q3i8_last_error(nullptr));
        }
        if (nr > 0) {
            const double t0 = now_ms();
            if ((rc = q3i8_cb_step(c, nr, r_slot.data(), r_pos.data(), r_tok.data(), out.data()))) return rc;
            decode_ms += now_ms() - t0;
            ++steps, step_rows += nr;
            if ((rc = q3i8_sched_complete_step(s, nr, out.data())))
                return fail(c, rc, "sched_run: %s", q3i8_last_error(nullptr));
        }
        if (na == 0 && nr == 0) return fail(c, Q3_ERR_STATE, "sched_run: the scheduler planned no work");
    }
    if (stats) {
        *stats = q3i8_stats{};
        stats->prefill_ms = prefill_ms, stats->decode_ms = decode_ms;
        stats->prefill_tokens = prefill_tokens, stats->decode_steps = steps;
        stats->prefill_tokens_per_sec = prefill_ms > 0 ? prefill_tokens / (prefill_ms * 1e-3) : 0;
        stats->decode_tokens_per_sec = decode_ms > 0 ? step_rows / (decode_ms * 1e-3) : 0;
        stats->step_us = steps > 0 ? decode_ms * 1e3 / steps : 0;
    }
    return Q3_OK;
}

extern "C" int q3i8_trace_step(q3i8_ctx* c, const int32_t* tokens, uint64_t* stamps, size_t cap, int32_t* grid,
                               int32_t* stride) {
    if (!c) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "ctx is NULL");
    if (c->active_B <= 0) return fail(c, Q3_ERR_STATE, "trace_step before q3i8_prefill");
    if (!persistent_for(c, c->active_B))
        return fail(c, Q3_ERR_STATE, "trace_step: this batch decodes with the chained step kernels");
    const int st = trace_stride(c->d.n_layers);
    const size_t n = (size_t)c->p_grid * st;
    if (grid) *grid = c->p_grid;
    if (stride) *stride = st;
    if (!stamps || !tokens || cap < n) return fail(c, Q3_ERR_STATE, "trace_step: need %zu stamps", n);
    const int B = c->active_B;
    for (int b = 0; b < B; ++b)
        if (c->seq_len[b] + 1 > c->cap) return fail(c, Q3_ERR_STATE, "sequence %d is at the context capacity", b);
    if (!c->p_trace) CK(c, cudaMalloc(&c->p_trace, n * 8));
    CK(c, cudaMemsetAsync(c->p_trace, 0, n * 8, c->stream));
    CK(c, cudaMemcpyAsync(c->tokens, tokens, B * 4, cudaMemcpyHostToDevice, c->stream));
    cudaError_t e = enqueue_persistent(c, B, nullptr, c->p_trace);
    if (e != cudaSuccess) return fail(c, Q3_ERR_CUDA, "trace_step launch: %s", cudaGetErrorString(e));
    c->launches += 1;
    CK(c, cudaMemcpyAsync(stamps, c->p_trace, n * 8, cudaMemcpyDeviceToHost, c->stream));
    int rc = check_status(c);
    if (rc) return rc;
    for (int b = 0; b < B; ++b) c->seq_len[b] += 1;
    return Q3_OK;
}

extern "C" int q3i8_read_kv(q3i8_ctx* c, int32_t layer, int32_t seq, int32_t n_pos, uint16_t* k, uint16_t* v) {
    if (!c) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "ctx is NULL");
    const q3i8_dims& d = c->d;
    if (layer < 0 || layer >= d.n_layers || seq < 0 || seq >= c->bmax || n_pos < 0 || n_pos > c->cap || !k || !v)
        return fail(c, Q3_ERR_INVALID_ARGUMENTS, "read_kv: argument out of range");
    CK(c, cudaStreamSynchronize(c->stream));
    const int hd = d.head_dim, nkv = d.n_kv_heads;
    for (int g = 0; g < nkv; ++g) {
        const size_t src = ((((size_t)layer * c->bmax + seq) * nkv + g) * c->cap) * hd;
        CK(c, cudaMemcpy(k + (size_t)g * n_pos * hd, c->kc + src, (size_t)n_pos * hd * 2, cudaMemcpyDeviceToHost));
        CK(c, cudaMemcpy(v + (size_t)g * n_pos * hd, c->vc + src, (size_t)n_pos * hd * 2, cudaMemcpyDeviceToHost));
    }
    return Q3_OK;
}

extern "C" int64_t q3i8_step_bytes(const q3i8_ctx* c, int32_t B, const int32_t* positions) {
    if (!c) return -1;
    const q3i8_dims& d = c->d;
    const int64_t H = d.hidden, I = d.intermediate, L = d.n_layers, hd = d.head_dim;
    const int64_t Dq = d.n_heads * hd, Dkv = d.n_kv_heads * hd;
    const int64_t w = (int64_t)d.vocab * H + L * ((Dq + 2 * Dkv) * H + H * Dq + 2 * I * H + H * I);
    const int64_t s = 4 * ((int64_t)d.vocab + L * ((Dq + 2 * Dkv) + H + 2 * I + H));
    const int64_t g = 4 * (L * (2 * H + 2 * hd) + H);
    int64_t kv = 0;
    for (int b = 0; b < B; ++b) kv += (int64_t)(positions ? positions[b] + 1 : 1) * L * 2 * Dkv * 2;
    kv += (int64_t)B * L * 2 * Dkv * 2;
    return w + s + g + kv;
}

extern "C" int32_t q3i8_step_launches(const q3i8_ctx* c, int32_t B) {
    return c ? step_launches(c, B) : 0;
}

extern "C" int64_t q3i8_launch_count(const q3i8_ctx* c) { return c ? c->launches : 0; }

extern "C" const char* q3i8_last_error(const q3i8_ctx* c) { return c ? c->err.c_str() : g_tls_error.c_str(); }

extern "C" const char* q3i8_status_name(int s) {
    switch (s) {
        case Q3_OK: return "ok";
        case Q3_ERR_UNSUPPORTED_ARCH: return "unsupported_architecture";
        case Q3_ERR_INVALID_ARGUMENTS: return "invalid_arguments";
        case Q3_ERR_CONTEXT: return "context_past_ceiling";
        case Q3_ERR_NO_DEVICE: return "no_device";
        case Q3_ERR_OOM: return "out_of_memory";
        case Q3_ERR_CUDA: return "cuda_error";
        case Q3_ERR_TIMEOUT: return "device_wait_timeout";
        case Q3_ERR_STATE: return "invalid_state";
        default: return "unknown_status";
    }
}

// ------------------------------------------------------------------ ops

extern "C" int q3i8_op_gemm_i8(const uint16_t* a_planes, const int8_t* w, const float* scale, int32_t M, int32_t N,
                               int32_t K, float* y, int32_t* d_status, void* cuda_stream) {
    if (!a_planes || !w || !scale || !y) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_gemm_i8: NULL pointer");
    if (M < 1 || !tc_gemm_supported(N, K))
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_gemm_i8: needs M >= 1, N %% 128 == 0, K %% 64 == 0");
    if (((uintptr_t)a_planes & 15) || ((uintptr_t)w & 15) || ((uintptr_t)y & 15))
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_gemm_i8: buffers must be 16-byte aligned");
    const int rc = launch_tc_gemm(reinterpret_cast<const __half*>(a_planes), w, scale, M, N, K, kStore, y, N, nullptr,
                                  0, d_status, (cudaStream_t)cuda_stream);
    if (rc) return fail(nullptr, Q3_ERR_CUDA, "op_gemm_i8: tensor-core GEMM could not be set up (%d)", rc);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(nullptr, Q3_ERR_CUDA, "op_gemm_i8 launch: %s", cudaGetErrorString(e));
    return Q3_OK;
}

static int current_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

extern "C" size_t q3i8_op_gemm_i8_splitk_workspace(int32_t M, int32_t N, int32_t K) {
    if (M < 1 || !tc_gemm_supported(N, K)) return 0;
    return tc_gemm_work_bytes(M, N, K, current_sms());
}

extern "C" int q3i8_op_gemm_i8_splitk(const uint16_t* a_planes, const int8_t* w, const float* scale, int32_t M,
                                      int32_t N, int32_t K, float* y, void* workspace, size_t ws_bytes,
                                      int32_t* d_status, void* cuda_stream) {
    if (!a_planes || !w || !scale || !y) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_gemm_i8_splitk: NULL pointer");
    if (M < 1 || !tc_gemm_supported(N, K))
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_gemm_i8_splitk: needs M >= 1, N %% 128 == 0, K %% 64 == 0");
    if (((uintptr_t)a_planes & 15) || ((uintptr_t)w & 15) || ((uintptr_t)y & 15) || ((uintptr_t)workspace & 15))
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_gemm_i8_splitk: buffers must be 16-byte aligned");
    const int sms = current_sms();
    if (ws_bytes < tc_gemm_work_bytes(M, N, K, sms) || (!workspace && tc_gemm_work_bytes(M, N, K, sms)))
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_gemm_i8_splitk: workspace too small");
    const int rc = launch_tc_gemm(reinterpret_cast<const __half*>(a_planes), w, scale, M, N, K, kStore, y, N, nullptr,
                                  0, d_status, (cudaStream_t)cuda_stream, (float*)workspace, ws_bytes, sms);
    if (rc) return fail(nullptr, Q3_ERR_CUDA, "op_gemm_i8_splitk: tensor-core GEMM could not be set up (%d)", rc);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(nullptr, Q3_ERR_CUDA, "op_gemm_i8_splitk launch: %s", cudaGetErrorString(e));
    return Q3_OK;
}

extern "C" size_t q3i8_op_attention_workspace(int32_t R, int32_t n_heads, int32_t hd, int32_t splits) {
    if (R <= 0 || n_heads <= 0 || hd <= 0 || splits <= 0) return 0;
    return attn_part_bytes(R, n_heads, hd, splits);
}

// Workspace of q3i8_op_sample: the settings, then the selection scratch.
static size_t op_sample_ws(int32_t B, int32_t V) {
    const size_t E = sample_band_entries(V);
    return 256 + (size_t)B * E * 8 + (size_t)B * E * 4;
}

extern "C" size_t q3i8_op_sample_workspace(int32_t B, int32_t V) {
    return (B < 1 || V < 1) ? 0 : op_sample_ws(B, V);
}

extern "C" int q3i8_op_sample(const float* logits, int32_t B, int32_t V, int32_t* counts,
                              const q3i8_sampling* sampling, int32_t step, int32_t* tokens, void* workspace,
                              size_t ws_bytes, int32_t* d_status, void* cuda_stream) {
    if (!logits || !counts || !tokens || !workspace || !sampling)
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_sample: NULL pointer");
    if (B < 1 || B > (1 << 20) || V < 1 || V > (1 << 28) || step < 0)
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_sample: unsupported sizes");
    bool greedy = false;
    if (validate_sampling(nullptr, sampling, &greedy)) return Q3_ERR_INVALID_ARGUMENTS;
    if (greedy) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_sample: temperature must be > 0");
    if (ws_bytes < op_sample_ws(B, V) || ((uintptr_t)workspace & 15))
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_sample: workspace too small or misaligned");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    const SampleParams p = device_params(*sampling);
    unsigned char* ws = (unsigned char*)workspace;
    cudaError_t e = cudaMemcpyAsync(ws, &p, sizeof p, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);  // p is a host temporary
    if (e != cudaSuccess) return fail(nullptr, Q3_ERR_CUDA, "op_sample: settings copy: %s", cudaGetErrorString(e));
    const size_t E = sample_band_entries(V);
    SampleArgs a{};
    a.logits = logits, a.ldz = V, a.V = V, a.counts = counts, a.params = (const SampleParams*)ws;
    a.step = nullptr, a.step_value = step, a.tokens = tokens, a.out_ids = nullptr, a.out_cap = 0;
    a.band_key = (uint64_t*)(ws + 256), a.band_tok = (int32_t*)(ws + 256 + (size_t)B * E * 8);
    a.status = d_status;
    e = launch_sample(a, B, st);
    if (e != cudaSuccess) return fail(nullptr, Q3_ERR_CUDA, "op_sample launch: %s", cudaGetErrorString(e));
    return Q3_OK;
}

extern "C" int q3i8_op_attention(const float* q, const uint16_t* k, const uint16_t* v, const int32_t* row_seq,
                                 const int32_t* row_len, int32_t R, int32_t n_heads, int32_t n_kv_heads, int32_t hd,
                                 int32_t cap, int32_t splits, float* out, void* workspace, size_t ws_bytes,
                                 int32_t* d_status, void* cuda_stream) {
    if (!q || !k || !v || !row_seq || !row_len || !out || !workspace)
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_attention: NULL pointer");
    if (R < 1 || n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || (hd != 64 && hd != 128) || cap < 64 ||
        cap % 64 || splits < 1 || splits > 64)
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_attention: unsupported sizes");
    if (ws_bytes < attn_part_bytes(R, n_heads, hd, splits) || ((uintptr_t)workspace & 15))
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_attention: workspace too small or misaligned");
    if (((uintptr_t)k & 15) || ((uintptr_t)v & 15))
        return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_attention: K/V caches must be 16-byte aligned");
    int rc = launch_attention(q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, row_seq, row_len, 0, R, n_heads,
                              n_kv_heads, hd, cap, splits, (float*)workspace, out, nullptr, 0, d_status,
                              (cudaStream_t)cuda_stream);
    if (rc) return fail(nullptr, Q3_ERR_INVALID_ARGUMENTS, "op_attention: unsupported head_dim/group");
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(nullptr, Q3_ERR_CUDA, "op_attention launch: %s", cudaGetErrorString(e));
    return Q3_OK;
}
