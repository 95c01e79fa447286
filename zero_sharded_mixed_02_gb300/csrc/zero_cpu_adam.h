// zero_cpu_adam.h -- the host side of ZeRO-Offload: Adam on host-resident fp32
// master, m and v from the 16-bit averaged gradient, and a small thread pool
// (host code only; built with the host compiler, no CUDA).
#pragma once

#include <condition_variable>
#include <cstdint>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

namespace zero {

// Everything one host Adam pass needs; constants derived from the
// hyperparameters once per step, as on the device.
struct HostAdamArgs {
    int dtype = 0;                  // 0 fp16, 1 bf16: the gradient and the params
    float loss_scale = 1.0f;        // the copied gradient is divided by it
    float clip_coef = 1.0f;
    float bc1 = 1.0f, bc2 = 1.0f;   // 1 - beta^t of this step
    float lr = 0.0f, beta1 = 0.0f, beta2 = 0.0f, eps = 0.0f, weight_decay = 0.0f;
    int decoupled_wd = 1;
};

// Elements [0, n) of the given arrays: master, m, v updated in place, params16
// written.  No threads; callers split the range.
void host_adam_range(const HostAdamArgs& a, const uint16_t* g16, float* master, float* m,
                     float* v, uint16_t* params16, int64_t n);

// A fixed set of worker threads running one task at a time: run(f) calls
// f(i, size) on every worker i (the calling thread is worker 0) and returns
// when all have finished.
class HostPool {
public:
    explicit HostPool(int size);
    ~HostPool();
    HostPool(const HostPool&) = delete;
    HostPool& operator=(const HostPool&) = delete;
    int size() const { return size_; }
    void run(const std::function<void(int, int)>& f);

private:
    void loop(int index);
    int size_ = 1;
    std::vector<std::thread> threads_;
    std::mutex mu_;
    std::condition_variable start_, done_;
    const std::function<void(int, int)>* task_ = nullptr;
    uint64_t generation_ = 0;
    int pending_ = 0;
    bool stop_ = false;
};

// Threads to use when the caller passes nthreads <= 0.
int host_threads_default();

}  // namespace zero
