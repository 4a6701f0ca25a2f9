// Quantized load cache ("Model-agnostic LLM inference", section "The
// quantized load cache"): one file holding the post-quantization bytes that
// q3i8_init takes (int8 weights, fp32 per-row scales, fp32 norm gains),
// behind a gate of magic + dims + SHA-256 of the caller's manifest + exact
// length.  A cache that fails the gate is reported, not used: the caller
// takes the full path and writes a fresh one.  Host code only.
//
// File layout (little-endian):
//   0    8  magic "Q3I8WC01"
//   8    4  format version (1)
//   12   4  header bytes (128)
//   16  44  dims: hidden, n_layers, n_heads, n_kv_heads, head_dim,
//           intermediate, vocab, rope_theta (f32 bits), rms_eps (f32 bits),
//           tie_word_embeddings, attention_bias
//   60  32  SHA-256 of the manifest bytes
//   92   8  payload bytes
//   100 28  zero
//   128     payload: embed w [V][H], embed scale [V], final_norm [H]; then per
//           layer q, k, v, o, gate, up, down (w, then scale) and attn_norm,
//           ffn_norm, q_norm, k_norm.
#include <errno.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#include <new>
#include <string>
#include <vector>

#include "../../include/q3i8.h"

int q3_report_error(int code, const char* msg);  // engine.cu

namespace {

// ------------------------------------------------------------------ SHA-256
// FIPS 180-4, section 6.2.  The round constants and the initial hash value
// are derived here from their definition (section 4.2.2 and 5.3.3): the
// first 32 bits of the fractional parts of the cube roots of the first 64
// primes and of the square roots of the first 8 primes.

typedef unsigned __int128 u128;

// floor(n^(1/k) * 2^32) for k = 2 or 3, by bisection on exact integers.
uint64_t root_fixed32(uint64_t n, int k) {
    const u128 target = (u128)n << (32 * k);
    uint64_t lo = 0, hi = (uint64_t)1 << 40;  // n < 2^9 so the root * 2^32 < 2^37
    while (lo < hi) {
        const uint64_t mid = lo + (hi - lo + 1) / 2;
        u128 p = (u128)mid * mid;
        if (k == 3) p *= mid;
        if (p <= target) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

struct ShaConstants {
    uint32_t k[64];
    uint32_t h0[8];
    ShaConstants() {
        int found = 0;
        for (uint64_t n = 2; found < 64; ++n) {
            bool prime = true;
            for (uint64_t d = 2; d * d <= n; ++d)
                if (n % d == 0) {
                    prime = false;
                    break;
                }
            if (!prime) continue;
            k[found] = (uint32_t)root_fixed32(n, 3);  // low 32 bits = fractional part
            if (found < 8) h0[found] = (uint32_t)root_fixed32(n, 2);
            ++found;
        }
    }
};

const ShaConstants& sha_constants() {
    static const ShaConstants c;
    return c;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

void sha256_block(uint32_t h[8], const uint8_t* p) {
    const ShaConstants& C = sha_constants();
    uint32_t w[64];
    for (int t = 0; t < 16; ++t)
        w[t] = (uint32_t)p[4 * t] << 24 | (uint32_t)p[4 * t + 1] << 16 | (uint32_t)p[4 * t + 2] << 8 | p[4 * t + 3];
    for (int t = 16; t < 64; ++t) {
        const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
        const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
        w[t] = w[t - 16] + s0 + w[t - 7] + s1;
    }
    uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
    for (int t = 0; t < 64; ++t) {
        const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
        const uint32_t ch = (e & f) ^ (~e & g);
        const uint32_t t1 = hh + S1 + ch + C.k[t] + w[t];
        const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
        const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
        const uint32_t t2 = S0 + maj;
        hh = g, g = f, f = e, e = d + t1, d = c, c = b, b = a, a = t1 + t2;
    }
    h[0] += a, h[1] += b, h[2] += c, h[3] += d, h[4] += e, h[5] += f, h[6] += g, h[7] += hh;
}

void sha256(const void* data, size_t len, uint8_t out[32]) {
    uint32_t h[8];
    memcpy(h, sha_constants().h0, sizeof h);
    const uint8_t* p = (const uint8_t*)data;
    size_t left = len;
    for (; left >= 64; left -= 64, p += 64) sha256_block(h, p);
    // padding (section 5.1.1): 0x80, zeros, the bit length as 64-bit big-endian
    uint8_t tail[128] = {0};
    memcpy(tail, p, left);
    tail[left] = 0x80;
    const size_t blocks = left + 9 <= 64 ? 1 : 2;
    const uint64_t bits = (uint64_t)len * 8;
    for (int i = 0; i < 8; ++i) tail[blocks * 64 - 1 - i] = (uint8_t)(bits >> (8 * i));
    for (size_t b = 0; b < blocks; ++b) sha256_block(h, tail + 64 * b);
    for (int i = 0; i < 8; ++i)
        for (int j = 0; j < 4; ++j) out[4 * i + j] = (uint8_t)(h[i] >> (24 - 8 * j));
}

// ------------------------------------------------------------------ layout

constexpr char kMagic[8] = {'Q', '3', 'I', '8', 'W', 'C', '0', '1'};
constexpr uint32_t kVersion = 1;
constexpr uint32_t kHeaderBytes = 128;
constexpr int kDimWords = 11;

void put_u32(uint8_t* p, uint32_t v) {
    for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
void put_u64(uint8_t* p, uint64_t v) {
    for (int i = 0; i < 8; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
uint32_t get_u32(const uint8_t* p) {
    uint32_t v = 0;
    for (int i = 0; i < 4; ++i) v |= (uint32_t)p[i] << (8 * i);
    return v;
}
uint64_t get_u64(const uint8_t* p) {
    uint64_t v = 0;
    for (int i = 0; i < 8; ++i) v |= (uint64_t)p[i] << (8 * i);
    return v;
}
uint32_t f32_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

void dim_words(const q3i8_dims& d, uint32_t w[kDimWords]) {
    w[0] = (uint32_t)d.hidden, w[1] = (uint32_t)d.n_layers, w[2] = (uint32_t)d.n_heads;
    w[3] = (uint32_t)d.n_kv_heads, w[4] = (uint32_t)d.head_dim, w[5] = (uint32_t)d.intermediate;
    w[6] = (uint32_t)d.vocab, w[7] = f32_bits(d.rope_theta), w[8] = f32_bits(d.rms_eps);
    w[9] = (uint32_t)d.tie_word_embeddings, w[10] = (uint32_t)d.attention_bias;
}

// The payload's arrays in file order; their sizes follow from the dims.
std::vector<size_t> piece_sizes(const q3i8_dims& d) {
    const size_t H = (size_t)d.hidden, I = (size_t)d.intermediate, V = (size_t)d.vocab;
    const size_t Dq = (size_t)d.n_heads * d.head_dim, Dkv = (size_t)d.n_kv_heads * d.head_dim;
    std::vector<size_t> s = {V * H, V * 4, H * 4};
    for (int l = 0; l < d.n_layers; ++l) {
        const size_t rows[7] = {Dq, Dkv, Dkv, H, I, I, H};
        const size_t cols[7] = {H, H, H, Dq, H, H, I};
        for (int m = 0; m < 7; ++m) s.push_back(rows[m] * cols[m]), s.push_back(rows[m] * 4);
        s.push_back(H * 4), s.push_back(H * 4), s.push_back((size_t)d.head_dim * 4), s.push_back((size_t)d.head_dim * 4);
    }
    return s;
}

uint64_t payload_bytes(const q3i8_dims& d) {
    uint64_t t = 0;
    for (size_t b : piece_sizes(d)) t += b;
    return t;
}

// The caller's arrays in file order (the same order as piece_sizes).
std::vector<const void*> piece_ptrs(const q3i8_mat* embed, const q3i8_layer* layers, const float* final_norm,
                                    int n_layers) {
    std::vector<const void*> p = {embed->w, embed->scale, final_norm};
    for (int l = 0; l < n_layers; ++l) {
        const q3i8_layer& L = layers[l];
        const q3i8_mat* m[7] = {&L.q, &L.k, &L.v, &L.o, &L.gate, &L.up, &L.down};
        for (int i = 0; i < 7; ++i) p.push_back(m[i]->w), p.push_back(m[i]->scale);
        p.push_back(L.attn_norm), p.push_back(L.ffn_norm), p.push_back(L.q_norm), p.push_back(L.k_norm);
    }
    return p;
}

int report(int code, const std::string& msg) { return q3_report_error(code, msg.c_str()); }

bool valid_dims(const q3i8_dims* dims, std::string* why) {
    char msg[512];
    if (q3i8_validate_dims(dims, msg, sizeof msg) != Q3_OK) {
        *why = msg;
        return false;
    }
    return true;
}

}  // namespace

struct q3i8_cache {
    q3i8_dims dims;
    std::vector<uint8_t> bytes;  // the whole file
    std::vector<q3i8_layer> layers;
    q3i8_mat embed;
    const float* final_norm;
};

extern "C" uint64_t q3i8_cache_payload_bytes(const q3i8_dims* dims) {
    if (!dims || dims->hidden <= 0 || dims->n_layers <= 0 || dims->n_heads <= 0 || dims->n_kv_heads <= 0 ||
        dims->head_dim <= 0 || dims->intermediate <= 0 || dims->vocab <= 0)
        return 0;
    return payload_bytes(*dims);
}

extern "C" int q3i8_cache_write(const char* path, const q3i8_dims* dims, const q3i8_mat* embed,
                                const q3i8_layer* layers, const float* final_norm, const void* manifest,
                                size_t manifest_len) {
    if (!path || !dims || !embed || !layers || !final_norm || (!manifest && manifest_len))
        return report(Q3_ERR_INVALID_ARGUMENTS, "cache_write: NULL argument");
    std::string why;
    if (!valid_dims(dims, &why)) return report(Q3_ERR_UNSUPPORTED_ARCH, "cache_write: " + why);
    const std::vector<size_t> sizes = piece_sizes(*dims);
    const std::vector<const void*> ptrs = piece_ptrs(embed, layers, final_norm, dims->n_layers);
    for (const void* p : ptrs)
        if (!p) return report(Q3_ERR_INVALID_ARGUMENTS, "cache_write: NULL weight, scale or gain pointer");

    uint8_t head[kHeaderBytes] = {0};
    memcpy(head, kMagic, 8);
    put_u32(head + 8, kVersion);
    put_u32(head + 12, kHeaderBytes);
    uint32_t w[kDimWords];
    dim_words(*dims, w);
    for (int i = 0; i < kDimWords; ++i) put_u32(head + 16 + 4 * i, w[i]);
    sha256(manifest ? manifest : "", manifest_len, head + 60);
    put_u64(head + 92, payload_bytes(*dims));

    // write beside the target, then rename: a reader never sees a partial file
    const std::string tmp = std::string(path) + ".tmp." + std::to_string((long long)getpid());
    FILE* f = fopen(tmp.c_str(), "wb");
    if (!f) return report(Q3_ERR_INVALID_ARGUMENTS, "cache_write: cannot create " + tmp + ": " + strerror(errno));
    bool ok = fwrite(head, 1, kHeaderBytes, f) == kHeaderBytes;
    for (size_t i = 0; ok && i < sizes.size(); ++i) ok = fwrite(ptrs[i], 1, sizes[i], f) == sizes[i];
    ok = (fclose(f) == 0) && ok;
    if (!ok || rename(tmp.c_str(), path) != 0) {
        const std::string err = strerror(errno);
        unlink(tmp.c_str());
        return report(Q3_ERR_INVALID_ARGUMENTS, std::string("cache_write: writing ") + path + " failed: " + err);
    }
    return Q3_OK;
}

extern "C" int q3i8_cache_open(const char* path, const q3i8_dims* dims, const void* manifest, size_t manifest_len,
                               q3i8_cache** out, int32_t* gate) {
    if (!path || !dims || !out || !gate || (!manifest && manifest_len))
        return report(Q3_ERR_INVALID_ARGUMENTS, "cache_open: NULL argument");
    *out = nullptr;
    *gate = Q3I8_CACHE_ABSENT;
    std::string why;
    if (!valid_dims(dims, &why)) return report(Q3_ERR_UNSUPPORTED_ARCH, "cache_open: " + why);

    FILE* f = fopen(path, "rb");
    if (!f) return Q3_OK;
    uint8_t head[kHeaderBytes];
    const size_t got = fread(head, 1, kHeaderBytes, f);
    if (got < 16 || memcmp(head, kMagic, 8) != 0 || get_u32(head + 8) != kVersion ||
        get_u32(head + 12) != kHeaderBytes) {
        fclose(f);
        *gate = Q3I8_CACHE_BAD_MAGIC;
        return Q3_OK;
    }
    if (got < kHeaderBytes) {
        fclose(f);
        *gate = Q3I8_CACHE_LENGTH;
        return Q3_OK;
    }
    uint32_t w[kDimWords];
    dim_words(*dims, w);
    for (int i = 0; i < kDimWords; ++i)
        if (get_u32(head + 16 + 4 * i) != w[i]) {
            fclose(f);
            *gate = Q3I8_CACHE_DIMS;
            return Q3_OK;
        }
    uint8_t digest[32];
    sha256(manifest ? manifest : "", manifest_len, digest);
    if (memcmp(head + 60, digest, 32) != 0) {
        fclose(f);
        *gate = Q3I8_CACHE_MANIFEST;
        return Q3_OK;
    }
    const uint64_t want = payload_bytes(*dims);
    if (fseeko(f, 0, SEEK_END) != 0) {
        fclose(f);
        return report(Q3_ERR_INVALID_ARGUMENTS, std::string("cache_open: cannot seek in ") + path);
    }
    const long long size = (long long)ftello(f);
    if (get_u64(head + 92) != want || size < 0 || (uint64_t)size != kHeaderBytes + want) {
        fclose(f);
        *gate = Q3I8_CACHE_LENGTH;
        return Q3_OK;
    }

    q3i8_cache* c = new (std::nothrow) q3i8_cache;
    if (!c) {
        fclose(f);
        return report(Q3_ERR_OOM, "cache_open: out of host memory");
    }
    try {
        c->bytes.resize((size_t)size);
    } catch (...) {
        fclose(f);
        delete c;
        return report(Q3_ERR_OOM, "cache_open: out of host memory for the payload");
    }
    const bool read_ok = fseeko(f, 0, SEEK_SET) == 0 && fread(c->bytes.data(), 1, (size_t)size, f) == (size_t)size;
    fclose(f);
    if (!read_ok) {
        delete c;
        *gate = Q3I8_CACHE_LENGTH;  // the file changed under us
        return Q3_OK;
    }
    // pointer tables into the payload, in file order
    c->dims = *dims;
    std::vector<const uint8_t*> at;
    const uint8_t* p = c->bytes.data() + kHeaderBytes;
    for (size_t b : piece_sizes(*dims)) at.push_back(p), p += b;
    size_t i = 0;
    c->embed.w = (const int8_t*)at[i++];
    c->embed.scale = (const float*)at[i++];
    c->final_norm = (const float*)at[i++];
    c->layers.resize(dims->n_layers);
    for (int l = 0; l < dims->n_layers; ++l) {
        q3i8_layer& L = c->layers[l];
        q3i8_mat* m[7] = {&L.q, &L.k, &L.v, &L.o, &L.gate, &L.up, &L.down};
        for (int k = 0; k < 7; ++k) m[k]->w = (const int8_t*)at[i++], m[k]->scale = (const float*)at[i++];
        L.attn_norm = (const float*)at[i++], L.ffn_norm = (const float*)at[i++];
        L.q_norm = (const float*)at[i++], L.k_norm = (const float*)at[i++];
    }
    *out = c;
    *gate = Q3I8_CACHE_VALID;
    return Q3_OK;
}

extern "C" int q3i8_cache_tables(const q3i8_cache* c, q3i8_mat* embed, q3i8_layer* layers, const float** final_norm) {
    if (!c || !embed || !layers || !final_norm) return report(Q3_ERR_INVALID_ARGUMENTS, "cache_tables: NULL argument");
    *embed = c->embed;
    for (int l = 0; l < c->dims.n_layers; ++l) layers[l] = c->layers[l];
    *final_norm = c->final_norm;
    return Q3_OK;
}

extern "C" void q3i8_cache_close(q3i8_cache* c) { delete c; }
