// zero_cpu_adam.cpp -- ZeRO-Offload's host Adam ([L18] sec. 4.4: the fp32
// master, m and v and the Adam update on the host, a multithreaded, vectorised
// host Adam; [ZL8] sec. 6.2, 7: the host runs the parameter update and sends
// the updated parameters back).
//
// Arithmetic: the same operations in the same order as the device update, each
// one binary32 rounding (the file is compiled with -ffp-contract=off, so no
// multiply-add is fused).  The element loop is branch-free so it vectorises
// (SSE on x86-64, Advanced SIMD on AArch64) without intrinsics.
#include "zero_cpu_adam.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>

#include "zero_b200.h"

namespace {

inline uint32_t f2u(float f)
{
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
}

inline float u2f(uint32_t u)
{
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// The two binary16 conversions below follow the published, public-domain
// bit-manipulation method for half-precision conversion described by Fabian
// "ryg" Giesen (his "half to float" / "float to half" routines and the write-up
// accompanying them, 2012-2013): widen by moving the exponent and fraction
// into place and rescaling with one exact multiplication; narrow by adding the
// exponent rebias and 0xFFF plus the kept bit's parity (round to nearest even),
// with subnormal results produced by the FPU through an added 0.5.  The code
// here is written from that description and tested exhaustively against the
// oracle's own conversions.
//
// binary16 -> binary32, exact.  The half's exponent and fraction bits moved up
// by 13 places, read as a binary32, are the half's value times 2^-112, for
// normal and subnormal halves alike (a half subnormal m 2^-24 becomes the
// binary32 subnormal m 2^-136); one multiplication by 2^112 is then exact.
// Exponent 31 (inf, NaN) gets the binary32 exponent 255, its fraction kept.
inline float half_to_float(uint16_t h)
{
    const uint32_t em = (uint32_t)(h & 0x7FFFu) << 13;
    uint32_t r = f2u(u2f(em) * 0x1p112f);
    r = em >= 0x0F800000u ? (r | 0x7F800000u) : r;
    return u2f(r | ((uint32_t)(h & 0x8000u) << 16));
}

// binary32 -> binary16, round to nearest even.  Results below 2^-14 come from
// adding 0.5 (whose ulp, 2^-24, is the binary16 subnormal step): the FPU's own
// rounding aligns the value, and the low bits are the code.  Normal results
// add the exponent rebias, 0xFFF and the kept bit's parity (ties to even) and
// shift out 13 bits; a carry into exponent 31 gives infinity.  |x| >= 2^16 is
// infinity; NaN becomes the quiet NaN 0x7E00 with the sign kept.
inline uint16_t float_to_half(float x)
{
    const uint32_t u = f2u(x);
    const uint32_t sign = (u >> 16) & 0x8000u;
    const uint32_t a = u & 0x7FFFFFFFu;
    const uint32_t normal = (a + 0xC8000FFFu + ((a >> 13) & 1u)) >> 13;
    const uint32_t sub = f2u(u2f(a) + 0.5f) - 0x3F000000u;
    const uint32_t special = a > 0x7F800000u ? 0x7E00u : 0x7C00u;
    const uint32_t r = a >= 0x47800000u ? special : (a < 0x38800000u ? sub : normal);
    return (uint16_t)(r | sign);
}

// bfloat16 is the upper half of binary32.
inline float bf16_to_float(uint16_t b) { return u2f((uint32_t)b << 16); }

// binary32 -> bfloat16, round to nearest even: add 0x7FFF plus the kept bit's
// parity, keep the upper half (a carry past the largest finite value gives
// infinity).  NaN becomes the quiet NaN 0x7FC0 with the sign kept.
inline uint16_t float_to_bf16(float x)
{
    const uint32_t u = f2u(x);
    const uint32_t r = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    const uint32_t nan = ((u >> 16) & 0x8000u) | 0x7FC0u;
    return (uint16_t)((u & 0x7FFFFFFFu) > 0x7F800000u ? nan : r);
}

struct Consts {
    float omb1, omb2, decay;
};

// The update works on blocks of BLOCK elements: widen the block's gradient into
// a small buffer, run Adam on binary32 values, narrow the updated master into
// the 16-bit parameters.  Three short loops keep each one's constants in
// registers (one fused loop ran 1.5x slower on Neoverse V2).
constexpr int64_t BLOCK = 1024;

template <int DT>
void widen_block(const uint16_t* __restrict in, float* __restrict out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = DT == 0 ? half_to_float(in[i]) : bf16_to_float(in[i]);
}

template <int DT>
void narrow_block(const float* __restrict in, uint16_t* __restrict out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = DT == 0 ? float_to_half(in[i]) : float_to_bf16(in[i]);
}

// WD: 0 none, 1 decoupled (AdamW: p *= 1 - lr wd), 2 L2 (g += wd p).
// POW2: the loss scale is a power of two whose reciprocal is a normal number,
// so dividing by it and multiplying by the reciprocal give the same result.
template <int WD, bool POW2>
void adam_block(const zero::HostAdamArgs& a, const Consts& k, const float* __restrict gw,
                float* __restrict master, float* __restrict m, float* __restrict v, int64_t n)
{
    const float S = a.loss_scale, inv_s = 1.0f / a.loss_scale;
    const float c = a.clip_coef, bc1 = a.bc1, bc2 = a.bc2;
    const float b1 = a.beta1, b2 = a.beta2, eps = a.eps, lr = a.lr, wd = a.weight_decay;
    const float omb1 = k.omb1, omb2 = k.omb2, decay = k.decay;
    for (int64_t i = 0; i < n; i++) {
        float g = POW2 ? gw[i] * inv_s : gw[i] / S;
        g = g * c;
        float p = master[i];
        if (WD == 1) p = p * decay;
        if (WD == 2) g = g + wd * p;
        const float mi = b1 * m[i] + omb1 * g;
        const float vi = b2 * v[i] + omb2 * (g * g);
        const float mhat = mi / bc1;
        const float vhat = vi / bc2;
        const float upd = mhat / (std::sqrt(vhat) + eps);
        p = p - lr * upd;
        master[i] = p;
        m[i] = mi;
        v[i] = vi;
    }
}

template <int DT, int WD, bool POW2>
void adam_range(const zero::HostAdamArgs& a, const Consts& k, const uint16_t* g16,
                float* master, float* m, float* v, uint16_t* out, int64_t n)
{
    alignas(64) float gw[BLOCK];
    for (int64_t b = 0; b < n; b += BLOCK) {
        const int64_t cnt = std::min(BLOCK, n - b);
        widen_block<DT>(g16 + b, gw, cnt);
        adam_block<WD, POW2>(a, k, gw, master + b, m + b, v + b, cnt);
        narrow_block<DT>(master + b, out + b, cnt);
    }
}

template <int DT, bool POW2>
void adam_dispatch_wd(const zero::HostAdamArgs& a, const Consts& k, const uint16_t* g16,
                      float* master, float* m, float* v, uint16_t* out, int64_t n)
{
    if (a.weight_decay == 0.0f) adam_range<DT, 0, POW2>(a, k, g16, master, m, v, out, n);
    else if (a.decoupled_wd) adam_range<DT, 1, POW2>(a, k, g16, master, m, v, out, n);
    else adam_range<DT, 2, POW2>(a, k, g16, master, m, v, out, n);
}

// +2^k with 2 <= biased exponent <= 252: 1/S is exactly 2^-k, a normal number
bool pow2_scale(float s)
{
    const uint32_t b = f2u(s);
    const uint32_t e = (b >> 23) & 0xFFu;
    return (b & 0x807FFFFFu) == 0 && e >= 2 && e <= 252;
}

}  // namespace

namespace zero {

void host_adam_range(const HostAdamArgs& a, const uint16_t* g16, float* master, float* m,
                     float* v, uint16_t* params16, int64_t n)
{
    Consts k{};
    k.omb1 = (float)(1.0 - (double)a.beta1);
    k.omb2 = (float)(1.0 - (double)a.beta2);
    k.decay = (float)(1.0 - (double)a.lr * (double)a.weight_decay);
    const bool p2 = pow2_scale(a.loss_scale);
    if (a.dtype == 0) {
        if (p2) adam_dispatch_wd<0, true>(a, k, g16, master, m, v, params16, n);
        else adam_dispatch_wd<0, false>(a, k, g16, master, m, v, params16, n);
    } else {
        if (p2) adam_dispatch_wd<1, true>(a, k, g16, master, m, v, params16, n);
        else adam_dispatch_wd<1, false>(a, k, g16, master, m, v, params16, n);
    }
}

HostPool::HostPool(int size) : size_(std::max(1, size))
{
    for (int i = 1; i < size_; i++) {
        try {
            threads_.emplace_back([this, i]() { loop(i); });
        } catch (...) {
            break;
        }
    }
    size_ = (int)threads_.size() + 1;
}

HostPool::~HostPool()
{
    {
        std::lock_guard<std::mutex> lk(mu_);
        stop_ = true;
    }
    start_.notify_all();
    for (auto& t : threads_) t.join();
}

void HostPool::loop(int index)
{
    uint64_t seen = 0;
    for (;;) {
        const std::function<void(int, int)>* task;
        {
            std::unique_lock<std::mutex> lk(mu_);
            start_.wait(lk, [&] { return stop_ || generation_ != seen; });
            if (stop_) return;
            seen = generation_;
            task = task_;
        }
        (*task)(index, size_);
        {
            std::lock_guard<std::mutex> lk(mu_);
            if (--pending_ == 0) done_.notify_one();
        }
    }
}

void HostPool::run(const std::function<void(int, int)>& f)
{
    {
        std::lock_guard<std::mutex> lk(mu_);
        task_ = &f;
        pending_ = size_ - 1;
        generation_++;
    }
    start_.notify_all();
    f(0, size_);
    std::unique_lock<std::mutex> lk(mu_);
    done_.wait(lk, [&] { return pending_ == 0; });
    task_ = nullptr;
}

int host_threads_default()
{
    const unsigned hw = std::thread::hardware_concurrency();
    return hw == 0 ? 4 : (int)std::min(hw, 64u);
}

}  // namespace zero

// ---- the C ABI entry point --------------------------------------------------
extern "C" zero_status_t zero_cpu_adam(const void* grads16, zero_dtype_t dtype, uint64_t n,
                                       float loss_scale, float clip_coef, float bc1, float bc2,
                                       const zero_hparams_t* hp, float* master, float* m,
                                       float* v, void* params16, int nthreads)
{
    if (dtype != ZERO_FP16 && dtype != ZERO_BF16) return ZERO_EINVAL;
    if (n == 0) return ZERO_OK;
    if (!grads16 || !hp || !master || !m || !v || !params16) return ZERO_EINVAL;
    if (!(loss_scale > 0.0f) || !(bc1 > 0.0f) || !(bc2 > 0.0f)) return ZERO_EINVAL;
    zero::HostAdamArgs a;
    a.dtype = (int)dtype;
    a.loss_scale = loss_scale;
    a.clip_coef = clip_coef;
    a.bc1 = bc1;
    a.bc2 = bc2;
    a.lr = hp->lr;
    a.beta1 = hp->beta1;
    a.beta2 = hp->beta2;
    a.eps = hp->eps;
    a.weight_decay = hp->weight_decay;
    a.decoupled_wd = hp->decoupled_wd;
    const int want = nthreads > 0 ? nthreads : zero::host_threads_default();
    // contiguous ranges of whole 64-element groups, one per thread
    const int64_t groups = (int64_t)((n + 63) / 64);
    const int t = (int)std::max<int64_t>(1, std::min<int64_t>(want, groups));
    const uint16_t* g = static_cast<const uint16_t*>(grads16);
    uint16_t* out = static_cast<uint16_t*>(params16);
    try {
        zero::HostPool pool(t);
        pool.run([&](int i, int size) {
            const int64_t lo = std::min<int64_t>((int64_t)n, groups * i / size * 64);
            const int64_t hi = std::min<int64_t>((int64_t)n, groups * (i + 1) / size * 64);
            if (hi > lo) zero::host_adam_range(a, g + lo, master + lo, m + lo, v + lo, out + lo, hi - lo);
        });
    } catch (...) {                             // allocation or thread start: nothing escapes
        return ZERO_ENOMEM;
    }
    return ZERO_OK;
}
