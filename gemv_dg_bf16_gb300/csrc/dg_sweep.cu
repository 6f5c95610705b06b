// dg_sweep.cu -- on-device sweep that writes the per-device shape table.
//
// mstar PR #1104, "What changed": one table per device; each entry keeps every
// candidate's time and parameters beside the choice; a size leaves the default
// only for a >= 2 % gain.  Strata PR #1297, "Summary": only variants that are
// byte-identical on device are tuned; "True-default baseline": the default
// candidate and the bitwise reference are the library's real no-table launch.
// "Decode optimization round 3", "Rejected paths": tuner-harness times disagree
// with in-context times, so candidates are timed exactly as the benchmark times
// calls (CUDA graphs of back-to-back calls over weight copies larger than L2).
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "dg_common.cuh"
#include "dg_internal.h"
#include "dg_rows.h"

namespace dg {
namespace {

__device__ __forceinline__ uint32_t mix(uint64_t i, uint32_t seed)
{
    uint64_t z = i * 0x9E3779B97F4A7C15ull + seed;
    z ^= z >> 31;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 29;
    return static_cast<uint32_t>(z >> 16);
}

// Uniform values in (-amp, amp) rounded to bf16.
__global__ void fill_bf16(uint16_t* p, size_t n, uint32_t seed, float amp)
{
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x) {
        const float u = (mix(i, seed) & 0xFFFFFF) * (1.0f / 16777216.0f) * 2.0f - 1.0f;
        p[i] = f32_to_bf16_bits(u * amp);
    }
}

// Random e4m3 codes without the two NaN codes.
__global__ void fill_e4m3(uint8_t* p, size_t n, uint32_t seed)
{
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x) {
        uint8_t c = static_cast<uint8_t>(mix(i, seed));
        if ((c & 0x7F) == 0x7F) c ^= 1;
        p[i] = c;
    }
}

__global__ void fill_f32(float* p, size_t n, uint32_t seed, float lo, float hi)
{
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x)
        p[i] = lo + (hi - lo) * ((mix(i, seed) & 0xFFFFFF) * (1.0f / 16777216.0f));
}

struct DevBuf {
    void* p = nullptr;
    size_t n = 0;
    ~DevBuf()
    {
        if (p) cudaFree(p);
    }
    bool alloc(size_t bytes)
    {
        n = bytes;
        return cudaMalloc(&p, bytes ? bytes : 16) == cudaSuccess;
    }
};

struct Cand {
    dg_choice c;
    float us = 0.0f;
    bool bitwise = false;
    bool ran = false;
};

bool same_choice(const dg_choice& a, const dg_choice& b)
{
    if (a.variant != b.variant) return false;
    for (int i = 0; i < 6; ++i)
        if (a.params[i] != b.params[i]) return false;
    return true;
}

dg_choice mk(int v, int p0, int p1 = 0, int p2 = 0, int p3 = 0)
{
    dg_choice c{};
    c.variant = v;
    c.params[0] = p0;
    c.params[1] = p1;
    c.params[2] = p2;
    c.params[3] = p3;
    return c;
}

// Candidates of the default's family (families never mix inside a bucket; the
// register-streamed and bulk-staged CUDA-core variants are one family).
std::vector<dg_choice> candidates(int op, const dg_choice& def)
{
    std::vector<dg_choice> out{def};
    auto add = [&](const dg_choice& c) {
        for (auto& o : out)
            if (same_choice(o, c)) return;
        out.push_back(c);
    };
    if (def.variant == DG_VAR_TC) {
        for (int st = 2; st <= 8; ++st) {
            dg_choice c = mk(DG_VAR_TC, st);
            c.params[1] = def.params[1];       // the K-split rule is part of the arithmetic
            add(c);
            if (op == DG_OP_GEMV_A8W8) {       // quantisation fused or in a launch of its own
                c.params[1] = 1 - def.params[1];
                add(c);
            }
        }
    } else if (def.variant == DG_VAR_MMA) {
        for (int ks : {0, 1, 2, 4, 8})
            for (int wpc : {0, 4, 8})
                for (int u : {0, 2, 4, 8}) {
                    if (wpc && ks > wpc) continue;
                    add(mk(DG_VAR_MMA, ks, wpc, 0, u));
                }
    } else if (op == DG_OP_MOE_W1 || op == DG_OP_MOE_W2) {
        const bool w1 = op == DG_OP_MOE_W1;
        for (int mt : {1, 2, 4})
            for (int wpc : {4, 8})
                for (int tile : {0, w1 ? 32 : 64, w1 ? 64 : 128}) {
                    dg_choice c = mk(DG_VAR_CC_WARP, 4, wpc, 0, tile);
                    c.params[4] = mt;
                    add(c);
                }
        // one row range of every expert per CTA: warps and CTAs per SM, pairs per pass
        for (int mt : {1, 2, 4})
            for (int wpc : {4, 8})
                for (int cps : {0, 1, 3}) {
                    dg_choice c = mk(DG_VAR_CC_WARP, 4, wpc, cps, 0);
                    c.params[4] = mt;
                    c.params[5] = kMoeOrderRange;
                    add(c);
                }
        // and the other order, whichever is the default
        for (int wpc : {4, 8}) {
            dg_choice c = mk(DG_VAR_CC_WARP, 4, wpc, 0, 0);
            c.params[4] = 2;
            c.params[5] = def.params[5] == kMoeOrderRange ? kMoeOrderUnits : kMoeOrderRange;
            add(c);
        }
    } else {
        for (int R : {1, 2, 4, 8})
            for (int wpc : {4, 8})
                for (int ks : {1, 2, 4}) {
                    if (op == DG_OP_GATE_UP_SILU && R < 2) continue;
                    add(mk(DG_VAR_CC_WARP, R, wpc, 0, ks > 1 ? ks : 0));
                }
        for (int cps : {1, 2})
            for (int st : {0, 4, 8}) add(mk(DG_VAR_CC_BULK, 0, st, cps));
    }
    return out;
}

struct Problem {
    int op, M, N, K, topk, E;
    std::vector<DevBuf> W;      // weight copies (rotated)
    DevBuf x, ids, gw, s, scale, out, out2, ws;
    size_t out_bytes = 0, out2_bytes = 0, ws_bytes = 0;
    int nrout = 1;              // MoE: routings rotated instead of weights
    std::vector<DevBuf> rids;

    dg_status call(const dg_choice& c, int rep, cudaStream_t st)
    {
        dg_stream_t s_ = reinterpret_cast<dg_stream_t>(st);
        const void* w = W[rep % W.size()].p;
        switch (op) {
        case DG_OP_GEMV_BF16:
            return dg_gemv_bf16(x.p, w, out.p, M, N, K, ws.p, ws_bytes, s_, &c);
        case DG_OP_GATE_UP_SILU:
            return dg_gate_up_silu(x.p, w, out.p, M, N, K, ws.p, ws_bytes, s_, &c);
        case DG_OP_HEAD_FP8_ARGMAX:
            return dg_head_fp8_argmax(x.p, w, static_cast<const float*>(scale.p), out.p,
                                      static_cast<int32_t*>(out2.p), M, N, K, ws.p, ws_bytes, s_, &c);
        case DG_OP_MOE_W1:
            return dg_moe_w1_silu(x.p, static_cast<const int32_t*>(rids[rep % nrout].p), w,
                                  static_cast<const float*>(s.p), out.p, M, topk, E, N, K, ws.p, ws_bytes, s_, &c);
        case DG_OP_MOE_W2:
            return dg_moe_w2(x.p, static_cast<const int32_t*>(rids[rep % nrout].p), static_cast<const float*>(gw.p),
                             w, static_cast<const float*>(s.p), out.p, M, topk, E, K, N, ws.p, ws_bytes, s_, &c);
        case DG_OP_GEMV_A8W8:
            return dg_gemv_a8w8_blockscale(x.p, w, static_cast<const float*>(s.p), out.p, M, N, K, ws.p, ws_bytes,
                                           s_, &c);
        default:
            return DG_ERR_INVALID_ARG;
        }
    }
};

dg_status check(cudaError_t e)
{
    if (e == cudaSuccess) return DG_OK;
    cudaGetLastError();
    return DG_ERR_CUDA;
}

dg_status setup(Problem& P, const DeviceInfo* dev)
{
    int l2 = 0;
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev->device);
    size_t wbytes = 0, xbytes = 0;
    const int M = P.M, N = P.N, K = P.K;
    switch (P.op) {
    case DG_OP_GEMV_BF16: wbytes = size_t(N) * K * 2; xbytes = size_t(M) * K * 2; P.out_bytes = size_t(M) * N * 2; break;
    case DG_OP_GATE_UP_SILU: wbytes = size_t(2) * N * K * 2; xbytes = size_t(M) * K * 2; P.out_bytes = size_t(M) * N * 2; break;
    case DG_OP_HEAD_FP8_ARGMAX:
        wbytes = size_t(N) * K; xbytes = size_t(M) * K * 2; P.out_bytes = size_t(M) * N * 2; P.out2_bytes = size_t(M) * 4;
        break;
    case DG_OP_MOE_W1:
        wbytes = size_t(P.E) * 2 * N * K; xbytes = size_t(M) * K * 2; P.out_bytes = size_t(M) * P.topk * N * 2; break;
    case DG_OP_MOE_W2:
        wbytes = size_t(P.E) * N * K; xbytes = size_t(M) * P.topk * K * 2; P.out_bytes = size_t(M) * N * 2; break;
    case DG_OP_GEMV_A8W8: wbytes = size_t(N) * K; xbytes = size_t(M) * K * 2; P.out_bytes = size_t(M) * N * 2; break;
    default: return DG_ERR_INVALID_ARG;
    }
    const bool moe = P.op == DG_OP_MOE_W1 || P.op == DG_OP_MOE_W2;
    size_t copies = moe ? 1 : std::max<size_t>(1, (3 * size_t(l2) + wbytes - 1) / std::max<size_t>(wbytes, 1));
    if (!moe && copies < 2 && wbytes < size_t(l2) * 3) copies = 2;
    P.W.resize(copies);
    for (size_t i = 0; i < copies; ++i) {
        if (!P.W[i].alloc(wbytes)) return DG_ERR_CUDA;
        if (P.op == DG_OP_GEMV_BF16 || P.op == DG_OP_GATE_UP_SILU)
            fill_bf16<<<1024, 256>>>(static_cast<uint16_t*>(P.W[i].p), wbytes / 2, 11, 1.0f / 32.0f);
        else
            fill_e4m3<<<1024, 256>>>(static_cast<uint8_t*>(P.W[i].p), wbytes, 13);
    }
    if (!P.x.alloc(xbytes)) return DG_ERR_CUDA;
    fill_bf16<<<256, 256>>>(static_cast<uint16_t*>(P.x.p), xbytes / 2, 17, 1.0f);
    if (!P.out.alloc(P.out_bytes) || !P.out2.alloc(P.out2_bytes ? P.out2_bytes : 16)) return DG_ERR_CUDA;
    P.ws_bytes = dg_workspace_bytes(static_cast<dg_op>(P.op), M, N, K, P.topk);
    if (!P.ws.alloc(P.ws_bytes)) return DG_ERR_CUDA;
    if (cudaMemset(P.ws.p, 0, P.ws_bytes) != cudaSuccess) return DG_ERR_CUDA;
    if (P.op == DG_OP_GEMV_A8W8) {
        const size_t nsc = size_t((N + 127) / 128) * ((K + 127) / 128);
        if (!P.s.alloc(nsc * 4)) return DG_ERR_CUDA;
        fill_f32<<<64, 256>>>(static_cast<float*>(P.s.p), nsc, 31, 1e-4f, 3e-4f);
    }
    if (P.op == DG_OP_HEAD_FP8_ARGMAX) {
        if (!P.scale.alloc(4)) return DG_ERR_CUDA;
        fill_f32<<<1, 32>>>(static_cast<float*>(P.scale.p), 1, 19, 1e-3f, 2e-3f);
    }
    if (moe) {
        const size_t srows = size_t(P.E) * (P.op == DG_OP_MOE_W1 ? 2 * N : N);
        if (!P.s.alloc(srows * 4)) return DG_ERR_CUDA;
        fill_f32<<<256, 256>>>(static_cast<float*>(P.s.p), srows, 23, 1e-3f, 2e-3f);
        if (!P.gw.alloc(size_t(M) * P.topk * 4)) return DG_ERR_CUDA;
        fill_f32<<<1, 256>>>(static_cast<float*>(P.gw.p), size_t(M) * P.topk, 29, 0.05f, 0.3f);
        P.nrout = 8;
        P.rids.resize(P.nrout);
        uint32_t st = 0x2545F491u;
        for (int r = 0; r < P.nrout; ++r) {
            std::vector<int32_t> ids(size_t(M) * P.topk);
            for (int t = 0; t < M; ++t)
                for (int k = 0; k < P.topk; ++k) {
                    int e;
                    bool dup;
                    do {
                        st ^= st << 13;
                        st ^= st >> 17;
                        st ^= st << 5;
                        e = static_cast<int>(st % static_cast<uint32_t>(P.E));
                        dup = false;
                        for (int j = 0; j < k; ++j) dup = dup || ids[size_t(t) * P.topk + j] == e;
                    } while (dup && P.topk <= P.E);
                    ids[size_t(t) * P.topk + k] = e;
                }
            if (!P.rids[r].alloc(ids.size() * 4)) return DG_ERR_CUDA;
            if (cudaMemcpy(P.rids[r].p, ids.data(), ids.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
                return DG_ERR_CUDA;
        }
    }
    return check(cudaDeviceSynchronize());
}

// Median microseconds per call of `c`, from graphs of `R` back-to-back calls.
dg_status time_choice(Problem& P, const dg_choice& c, int reps, float* us)
{
    const int R = 16;
    cudaStream_t st;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return check(cudaErrorUnknown);
    dg_status s = DG_OK;
    for (int i = 0; i < 2 && s == DG_OK; ++i) s = P.call(c, i, st);     // warm (host caches)
    if (s == DG_OK) s = check(cudaStreamSynchronize(st));
    cudaGraph_t g = nullptr;
    cudaGraphExec_t ge = nullptr;
    if (s == DG_OK) {
        s = check(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
        if (s == DG_OK) {
            for (int i = 0; i < R && s == DG_OK; ++i) s = P.call(c, i, st);
            const dg_status e = check(cudaStreamEndCapture(st, &g));
            if (s == DG_OK) s = e;
        }
    }
    if (s == DG_OK) s = check(cudaGraphInstantiate(&ge, g, 0));
    std::vector<float> t;
    if (s == DG_OK) {
        cudaEvent_t e0, e1;
        cudaEventCreate(&e0);
        cudaEventCreate(&e1);
        for (int i = 0; i < 3 && s == DG_OK; ++i) s = check(cudaGraphLaunch(ge, st));
        for (int i = 0; i < reps && s == DG_OK; ++i) {
            cudaEventRecord(e0, st);
            s = check(cudaGraphLaunch(ge, st));
            cudaEventRecord(e1, st);
            if (s == DG_OK) s = check(cudaEventSynchronize(e1));
            float ms = 0.0f;
            cudaEventElapsedTime(&ms, e0, e1);
            t.push_back(ms * 1000.0f / R);
        }
        cudaEventDestroy(e0);
        cudaEventDestroy(e1);
    }
    if (ge) cudaGraphExecDestroy(ge);
    if (g) cudaGraphDestroy(g);
    cudaStreamDestroy(st);
    if (s != DG_OK) return s;
    std::sort(t.begin(), t.end());
    *us = t.empty() ? 0.0f : t[t.size() / 2];
    return DG_OK;
}

// One call on weight copy 0, then the output bytes.
dg_status run_once(Problem& P, const dg_choice& c, std::vector<uint8_t>& bytes)
{
    dg_status s = P.call(c, 0, nullptr);
    if (s != DG_OK) return s;
    if ((s = check(cudaDeviceSynchronize())) != DG_OK) return s;
    bytes.resize(P.out_bytes + P.out2_bytes);
    if ((s = check(cudaMemcpy(bytes.data(), P.out.p, P.out_bytes, cudaMemcpyDeviceToHost))) != DG_OK) return s;
    if (P.out2_bytes)
        s = check(cudaMemcpy(bytes.data() + P.out_bytes, P.out2.p, P.out2_bytes, cudaMemcpyDeviceToHost));
    return s;
}

std::string choice_json(const dg_choice& c)
{
    char b[160];
    std::snprintf(b, sizeof b, "{\"variant\": %d, \"params\": [%d, %d, %d, %d, %d, %d]}", c.variant, c.params[0],
                  c.params[1], c.params[2], c.params[3], c.params[4], c.params[5]);
    return b;
}

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" dg_status dg_sweep(const dg_shape* shapes, int n_shapes, const char* out_path, int reps)
{
    if (!shapes || n_shapes < 1 || !out_path) return DG_ERR_INVALID_ARG;
    if (reps < 3) reps = 3;
    dg_status s;
    const DeviceInfo* dev = current_device(&s);
    if (!dev) return s;
    std::string entries;
    dg_status first_err = DG_OK;
    for (int i = 0; i < n_shapes && first_err == DG_OK; ++i) {
        Problem P;
        P.op = shapes[i].op;
        P.M = shapes[i].M;
        P.N = shapes[i].N;
        P.K = shapes[i].K;
        P.topk = shapes[i].topk;
        P.E = shapes[i].E > 0 ? shapes[i].E : 128;
        const int bucket = bucket_rows(P.M);
        if (P.op < 0 || P.op >= DG_OP_COUNT || bucket < 0 || P.N < 1 || P.K < 1) {
            first_err = DG_ERR_INVALID_ARG;
            break;
        }
        if ((s = setup(P, dev)) != DG_OK) {
            first_err = s;
            break;
        }
        dg_choice def;
        default_choice(static_cast<dg_op>(P.op), bucket, P.N, P.K, &def);
        std::vector<Cand> cands;
        for (const auto& c : candidates(P.op, def)) cands.push_back(Cand{c});
        std::vector<uint8_t> ref, got;
        if ((s = run_once(P, def, ref)) != DG_OK) {
            first_err = s;
            break;
        }
        for (auto& cd : cands) {
            if (run_once(P, cd.c, got) != DG_OK) continue;      // candidate does not fit this shape
            cd.bitwise = (got == ref);
            if (time_choice(P, cd.c, reps, &cd.us) != DG_OK) continue;
            cd.ran = true;
        }
        const Cand& d = cands[0];
        if (!d.ran) {
            first_err = DG_ERR_CUDA;
            break;
        }
        const Cand* pick = &d;
        for (const auto& cd : cands)
            if (cd.ran && cd.bitwise && cd.us < pick->us) pick = &cd;
        if (pick->us > 0.98f * d.us) pick = &d;                 // keep the default unless >= 2 % faster
        float pick_us = pick->us, def_us = d.us;
        if (pick != &d) {
            // Confirm: the default and the pick timed alternately three more times each;
            // the pick stays only if its median is still >= 2 % below the default's
            // (one timing's spread is about that much, so a single win can be noise).
            std::vector<float> td, tp;
            for (int r = 0; r < 3; ++r) {
                float u = 0.0f;
                if (time_choice(P, d.c, reps, &u) == DG_OK) td.push_back(u);
                if (time_choice(P, pick->c, reps, &u) == DG_OK) tp.push_back(u);
            }
            if (td.size() == 3 && tp.size() == 3) {
                std::sort(td.begin(), td.end());
                std::sort(tp.begin(), tp.end());
                def_us = td[1];
                pick_us = tp[1];
            }
            if (td.size() != 3 || tp.size() != 3 || pick_us > 0.98f * def_us) {
                pick = &d;
                pick_us = def_us;
            }
        }
        char head[256];
        std::snprintf(head, sizeof head, "    {\"op\": \"%s\", \"M\": %d, \"N\": %d, \"K\": %d, ", op_key_name(P.op),
                      bucket, P.N, P.K);
        std::string e = head;
        e += "\"pick\": " + choice_json(pick->c);
        char b[128];
        std::snprintf(b, sizeof b, ", \"pick_us\": %.3f, ", pick_us);
        e += b;
        e += "\"default\": " + choice_json(d.c);
        std::snprintf(b, sizeof b, ", \"default_us\": %.3f, \"candidates\": [", def_us);
        e += b;
        bool first = true;
        for (const auto& cd : cands) {
            if (!cd.ran) continue;
            e += first ? "" : ", ";
            first = false;
            std::snprintf(b, sizeof b, "{\"variant\": %d, \"params\": [%d, %d, %d, %d, %d, %d], \"us\": %.3f, \"bitwise\": %s}",
                          cd.c.variant, cd.c.params[0], cd.c.params[1], cd.c.params[2], cd.c.params[3],
                          cd.c.params[4], cd.c.params[5], cd.us, cd.bitwise ? "true" : "false");
            e += b;
        }
        e += "]}";
        if (!entries.empty()) entries += ",\n";
        entries += e;
    }
    if (first_err != DG_OK) return first_err;
    FILE* f = std::fopen(out_path, "w");
    if (!f) return DG_ERR_INVALID_ARG;
    std::fprintf(f,
                 "{\n  \"format\": \"libdecodegemm-table\",\n  \"identity\": {\"arch\": \"sm_%d%d\", \"driver\": %d, "
                 "\"runtime\": %d, \"build\": \"%s\", \"selection_space\": %d, \"device\": \"%s\"},\n"
                 "  \"entries\": [\n%s\n  ]\n}\n",
                 dev->cc_major, dev->cc_minor, dev->driver_version, dev->runtime_version, build_id(),
                 dg_selection_space(), dev->name, entries.c_str());
    std::fclose(f);
    return DG_OK;
}
