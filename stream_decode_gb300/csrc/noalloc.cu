// noalloc.cu -- gpt2_cached_step_noalloc: one cached decode step that
// allocates no device memory.
//
// Who needs it: callers that may not allocate device memory while they run
// steps.  Some host frameworks own every device allocation themselves (a
// plug-in or an embedded runtime with a fixed, pre-reserved memory budget).
// Some latency-critical loops cannot afford cudaMalloc, which may
// synchronise the device and has no latency bound.  Such a caller creates
// the model once at start-up, keeps its own KV-cache, logits and token
// buffers, and steps with this entry point, which needs nothing else.
//
// The step kernel's scratch (activation vectors, attention partials, greedy
// partials as tagged exchange words, status words) lives in the file-scope
// array `g_step_scratch` below, of kScratchMax bytes; every GPU that loads
// the library holds that array until the process exits.  Host code may not
// pass the symbol itself to a kernel: on the host it names a stand-in, not
// the device array, so a kernel given it would fault or, where the GPU can
// reach host memory, silently use the wrong memory.  The device address is
// fetched once per device with cudaGetSymbolAddress, with that device
// current: gpt2_model_create does it (noalloc_prepare), which also makes
// CUDA load this module and its array there even under lazy module loading,
// so stepping itself does no set-up; a call on a device where no model was
// created does the set-up on its first call.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "../../include/gpt2.h"
#include "gpt2_dev.cuh"
#include "model_internal.h"

namespace gpt2 {
cudaError_t launch_step(const StepPlan& P, int wq, cudaStream_t stream);
cudaError_t launch_cstep(const CPlan& P, int wf, cudaStream_t stream);
}

using namespace gpt2;

namespace {

// Largest scratch one call may use (GPT-2 124M needs about 360 KB on the
// cluster step kernel, 70 KB on the per-phase kernel).
constexpr size_t kScratchMax = 512 * 1024;
constexpr int kMaxDevices = 64;
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __align__(256) unsigned char g_step_scratch[kScratchMax];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_step_scratch on the current device (set up once per device).
gpt2_status scratch_base(unsigned char** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return GPT2_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GPT2_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_step_scratch);
        if (e != cudaSuccess || !p) return GPT2_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<unsigned char*>(g_scratch_addr[dev]);
    return GPT2_OK;
}

}  // namespace

namespace gpt2 {
// Set-up of the scratch array on the current device (called by gpt2_model_create).
bool noalloc_prepare() {
    unsigned char* base = nullptr;
    return scratch_base(&base) == GPT2_OK;
}
}  // namespace gpt2

extern "C" gpt2_status gpt2_cached_step_noalloc(const gpt2_model* m, float* d_cache, uint32_t position,
                                                uint32_t token, float* d_logits, uint32_t* d_next_token,
                                                void* stream) {
    if (!m || !d_cache) return GPT2_ERR_ARG;
    const gpt2_config& c = m->cfg;
    if (token >= c.vocab) return GPT2_ERR_TOKEN;
    if (position >= c.max_pos) return GPT2_ERR_POSITION;
    const ScratchLayout k = scratch_layout((int)c.d_model, (int)c.n_head, (int)c.d_ff, m->G);
    const CScratch ck = cscratch_layout((int)c.d_model, (int)c.n_head, m->cg.NC, m->cg.G);
    const size_t need = m->ckern ? ck.total : k.total;
    if (need > kScratchMax) return GPT2_ERR_SCRATCH;
    unsigned char* base = nullptr;
    gpt2_status st = scratch_base(&base);
    if (st != GPT2_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // The array keeps the previous call's contents.  Every call numbers its
    // phases from the same start, so the status words and every tagged
    // exchange word must start at zero (no stale tag may match); the greedy
    // history starts empty.
    cudaError_t e = cudaMemsetAsync(base, 0, need, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(base + (m->ckern ? ck.last_token : k.last_token), 0xFF, 8, s);
    if (e == cudaSuccess && d_next_token) e = cudaMemsetAsync(d_next_token, 0xFF, 4, s);
    if (e != cudaSuccess) return GPT2_ERR_CUDA;

    StepPlan P;
    memset(&P, 0, sizeof(P));
    P.L = (int)c.n_layer;
    P.D = (int)c.d_model;
    P.H = (int)c.n_head;
    P.FF = (int)c.d_ff;
    P.V = (int)c.vocab;
    P.n_pos = (int)c.n_pos;
    P.max_pos = (int)c.max_pos;
    P.G = m->G;
    P.packed = m->d_packed;
    P.fold = m->d_fold;
    P.wstream = m->d_wstream;
    P.layer_bytes = m->layer_bytes;
    for (int i = 0; i < 4; ++i) P.mat_off[i] = m->mat_off[i];
    P.vocab = m->wfmt != kWF32 ? m->d_vocab : reinterpret_cast<const uint8_t*>(m->d_packed + m->wte_off);
    P.wte_off = m->wte_off;
    P.wpe_off = m->wpe_off;
    P.lnf_g = m->lnf_g;
    P.lnf_b = m->lnf_b;
    for (uint32_t l = 0; l < c.n_layer; ++l) P.lp[l] = m->lp[l];
    P.cache = d_cache;
    P.xa = reinterpret_cast<uint64_t*>(base + k.xa);
    P.xb = reinterpret_cast<uint64_t*>(base + k.xb);
    P.qkv = reinterpret_cast<uint64_t*>(base + k.qkv);
    P.u = reinterpret_cast<uint64_t*>(base + k.u);
    P.attn_part = reinterpret_cast<uint64_t*>(base + k.attn);
    P.arg_part = reinterpret_cast<uint64_t*>(base + k.arg);
    P.status = reinterpret_cast<int*>(base + k.words);
    P.abort_flag = reinterpret_cast<int*>(base + k.words) + 1;
    P.last_token = reinterpret_cast<uint32_t*>(base + k.last_token);
    P.epoch = 0;
    P.p0 = (int)position;
    P.n_steps = 1;
    P.tokens_in = nullptr;
    P.token0 = token;
    P.tokens_out = d_next_token;
    P.logits = d_logits;
    P.logits_stride = 0;
    P.trace = nullptr;
    P.wait_limit_ns = kWaitNs;
    P.stall_phase = -1;
    P.prefetch_chunks = 0;
    P.pace_ns = kDefaultPaceNs;
    P.act_row = m->quant == GPT2_INT8_ROW_ACT;
    if (m->ckern) {
        // the cluster step kernel: the same plan, its geometry and exchange words
        CPlan C;
        memset(&C, 0, sizeof(C));
        C.s = P;
        C.g = m->cg;
        C.cstream = m->d_cstream;
        C.partO = reinterpret_cast<uint64_t*>(base + ck.partO);
        C.partP = reinterpret_cast<uint64_t*>(base + ck.partP);
        C.s.xa = C.s.xb = C.s.qkv = C.s.u = C.s.attn_part = nullptr;
        C.s.arg_part = reinterpret_cast<uint64_t*>(base + ck.arg);
        C.s.status = reinterpret_cast<int*>(base + ck.words);
        C.s.abort_flag = reinterpret_cast<int*>(base + ck.words) + 1;
        C.s.last_token = reinterpret_cast<uint32_t*>(base + ck.last_token);
        e = launch_cstep(C, m->wfmt, s);
    } else {
        e = launch_step(P, m->wfmt, s);
    }
    return e == cudaSuccess ? GPT2_OK : (e == cudaErrorMemoryAllocation ? GPT2_ERR_NOMEM : GPT2_ERR_CUDA);
}
