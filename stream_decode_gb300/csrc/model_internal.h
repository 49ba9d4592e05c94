// model_internal.h -- the device-resident model handle shared by the
// library's translation units.
#pragma once
#include <cstdint>

#include "../../include/gpt2.h"
#include "cstep.cuh"
#include "gpt2_dev.cuh"

struct gpt2_model {
    gpt2_config cfg;
    int quant;  // gpt2_quant of the model
    int wfmt;   // weight format of the device streams (kWF32, kWQ8, kWF16)
    int G;
    float* d_packed;
    uint8_t* d_wstream;
    uint8_t* d_vocab;  // int8 and binary16 models: the tied embedding's rows in the model's weight format
    uint64_t layer_bytes;
    uint64_t mat_off[4];
    uint64_t wte_off, wpe_off, lnf_g, lnf_b;
    gpt2::LayerParams lp[gpt2::kMaxLayers];
    float* d_fold;  // binary32 models: LayerNorm folds of the QKV and FC rows (fold_layer_words per layer)
    float* d_wlo;  // binary32 models: TF32 remainders of the block matrices (prefill), made on first use
    float* d_wte_lo;  // binary32 models: TF32 remainders of the tied embedding (batched decode), made on first use
    int ckern;        // 1: decode steps run on the cluster step kernel (cstep.cu), 0: on step_kernel (decode.cu)
    gpt2::CGeo cg;    // its geometry
    uint8_t* d_cstream;  // its weight stream
};
