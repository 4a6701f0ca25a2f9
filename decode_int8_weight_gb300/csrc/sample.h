// The seeded sampling chain on the device (host side of sample.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace q3 {

constexpr int kSampleMaxTopK = 4096;     // candidates held (and sorted) in shared memory
constexpr int kSampleCtas = 8;           // CTAs (one cluster) per sequence
constexpr int kStatusSampleSelect = 9;   // the top-k selection did not add up (an internal error)

// Settings of the chain ("Model-agnostic LLM inference", section
// "Sampling"), in device memory so that a captured step graph reads them at
// every replay.
struct SampleParams {
    double temperature;        // > 0
    double top_p;              // (0, 1]
    double min_p;              // [0, 1]
    double repeat_penalty;     // > 0 (1: off)
    double presence_penalty;
    double frequency_penalty;
    int32_t top_k;             // 1 .. kSampleMaxTopK
    int32_t pad;
    uint64_t seed;
};

struct SampleArgs {
    const float* logits;       // [B][ldz] this step's logits
    int ldz, V;
    int32_t* counts;           // [B][V] occurrences of each token in the sequence so far (updated)
    const SampleParams* params;
    const int32_t* step;       // device counter: the draw is for generated token *step - 1 (NULL: step_value)
    int step_value;
    int32_t* tokens;           // [B] the drawn token
    int32_t* out_ids;          // [B][out_cap] (may be NULL): column *step - 1 receives the token
    int out_cap;
    uint64_t* band_key;        // [B][sample_band_entries(V)] scratch
    int32_t* band_tok;         // [B][sample_band_entries(V)] scratch
    int32_t* status;           // set to kStatusSampleSelect if the selection is inconsistent (may be NULL)
};

// Scratch entries per sequence of the band lists.
size_t sample_band_entries(int V);

// One cluster of kSampleCtas CTAs per sequence: penalties -> temperature ->
// top-k -> min-p -> top-p -> the seeded draw; writes the token and counts it.
cudaError_t launch_sample(const SampleArgs& a, int B, cudaStream_t st);

// counts[row_seq[m]][ids[m]] += 1 for the m < M prompt rows.
cudaError_t launch_count_tokens(const int32_t* ids, const int32_t* row_seq, int M, int32_t* counts, int V,
                                cudaStream_t st);

}  // namespace q3
