// profile.cu -- optional per-launch CUDA-event timing (see dspark_profile_* in dspark.h).
#include <cuda_runtime.h>

#include <vector>

#include "common.cuh"
#include "profile.h"

namespace dspark {

namespace {
struct Rec {
    int name;
    cudaEvent_t a, b;
};
bool g_on = false;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;
int g_open = -1;

const char* const kNames[] = {"draft_prep",      "draft_sweep_generic", "draft_sweep_tc",   "verify_pass1",
                              "verify_accept",   "verify_residual_generic", "verify_residual_tc",
                              "verify_sample",   "schedule",            "draft_prep_rnn",   "draft_rnn_gru",
                              "schedule_threshold", "sts_hist",           "sts_ece",          "sts_advance",
                              "sts_apply",          "sts_fix",
                              "draft_rnn_gru_finish"};

cudaEvent_t take() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}
}  // namespace

void prof_begin(int name, cudaStream_t s) {
    if (!g_on) return;
    Rec r{name, take(), take()};
    cudaEventRecord(r.a, s);
    g_recs.push_back(r);
    g_open = (int)g_recs.size() - 1;
}

void prof_end(cudaStream_t s) {
    if (!g_on || g_open < 0) return;
    cudaEventRecord(g_recs[g_open].b, s);
    g_open = -1;
}

}  // namespace dspark

using namespace dspark;

extern "C" {

int dspark_profile_enable(int on) {
    g_on = on != 0;
    return DSPARK_OK;
}

int dspark_profile_collect(int32_t* name_ids, float* ms, int cap) {
    const int n = (int)g_recs.size();
    int st = DSPARK_OK;
    for (int i = 0; i < n; ++i) {
        Rec& r = g_recs[i];
        float t = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
            st = DSPARK_ERR_CUDA;
        if (i < cap) {
            if (name_ids) name_ids[i] = r.name;
            if (ms) ms[i] = t;
        }
        g_pool.push_back(r.a);
        g_pool.push_back(r.b);
    }
    g_recs.clear();
    g_open = -1;
    return st == DSPARK_OK ? n : st;
}

const char* dspark_profile_kernel_name(int name_id) {
    const int n = (int)(sizeof(kNames) / sizeof(kNames[0]));
    return (name_id >= 0 && name_id < n) ? kNames[name_id] : "unknown";
}

}  // extern "C"
