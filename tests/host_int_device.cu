// Host build of the scalar integer routines of the kernels' device header
// (int_device.cuh). Reads input arrays from DIR, writes the routines'
// outputs beside them; tests/test_int_device_host.py compares them with the
// oracle. Files are raw little-endian arrays: <name>.bin.
#include <stdio.h>
#include <stdlib.h>
#include <string>
#include <vector>
#include "../deterministic_integer_only_gb300/csrc/int_device.cuh"

using namespace detint;

template <class T>
static std::vector<T> load(const std::string& dir, const char* name) {
    std::vector<T> v;
    FILE* f = fopen((dir + "/" + name + ".bin").c_str(), "rb");
    if (!f) { fprintf(stderr, "missing %s\n", name); exit(2); }
    fseek(f, 0, SEEK_END);
    const long n = ftell(f) / (long)sizeof(T);
    fseek(f, 0, SEEK_SET);
    v.resize(n);
    if (n && fread(v.data(), sizeof(T), n, f) != (size_t)n) exit(2);
    fclose(f);
    return v;
}

template <class T>
static void save(const std::string& dir, const char* name, const std::vector<T>& v) {
    FILE* f = fopen((dir + "/" + name + ".bin").c_str(), "wb");
    if (!f) exit(3);
    if (!v.empty()) fwrite(v.data(), sizeof(T), v.size(), f);
    fclose(f);
}

int main(int argc, char** argv) {
    if (argc < 2) return 1;
    const std::string dir = argv[1];
    {   // rounding shift
        auto x = load<i64>(dir, "rshr_x");
        auto s = load<int32_t>(dir, "rshr_s");
        std::vector<i64> out(x.size());
        for (size_t i = 0; i < x.size(); ++i) out[i] = rshr(x[i], s[i]);
        save(dir, "rshr_out", out);
    }
    {   // floor square root
        auto x = load<u64>(dir, "isqrt_x");
        std::vector<u64> out(x.size());
        for (size_t i = 0; i < x.size(); ++i) out[i] = isqrt_u64(x[i]);
        save(dir, "isqrt_out", out);
        auto xf = load<u64>(dir, "isqrtf_x");
        std::vector<u64> of(xf.size());
        for (size_t i = 0; i < xf.size(); ++i) of[i] = isqrt_fast(xf[i]);
        save(dir, "isqrtf_out", of);
    }
    {   // 15-bit dyadic scale
        auto N = load<u64>(dir, "dyadic_n");
        auto D = load<u64>(dir, "dyadic_d");
        std::vector<int32_t> m(N.size()), k(N.size());
        for (size_t i = 0; i < N.size(); ++i) {
            int mm, kk;
            dyadic_dev(N[i], D[i], &mm, &kk);
            m[i] = mm;
            k[i] = kk;
        }
        save(dir, "dyadic_m", m);
        save(dir, "dyadic_k", k);
    }
    {   // 2^(delta/1024) in Q15
        auto d = load<i64>(dir, "exp2q_d");
        std::vector<i64> out(d.size());
        for (size_t i = 0; i < d.size(); ++i) out[i] = exp2q_dev(d[i]);
        save(dir, "exp2q_out", out);
    }
    {   // SwiGLU channel
        auto g = load<int32_t>(dir, "swiglu_g");
        auto u = load<int32_t>(dir, "swiglu_u");
        std::vector<int32_t> out(g.size());
        for (size_t i = 0; i < g.size(); ++i) out[i] = swiglu_dev(g[i], u[i]);
        save(dir, "swiglu_out", out);
    }
    {   // dyadic scales by the single-thread Newton-Raphson form
        auto n = load<u64>(dir, "dyadic_n");
        auto dd = load<u64>(dir, "dyadic_d");
        std::vector<int32_t> mo(n.size()), ko(n.size());
        for (size_t i = 0; i < n.size(); ++i) dyadic_fast(n[i], dd[i], &mo[i], &ko[i]);
        save(dir, "dyadicf_m", mo);
        save(dir, "dyadicf_k", ko);
    }
    {   // exact-mode requantisation: rshr(acc * M, s) through a 128-bit product
        auto acc = load<i64>(dir, "mul128_acc");
        auto M = load<u64>(dir, "mul128_m");
        auto sh = load<int32_t>(dir, "mul128_s");
        std::vector<i64> out(acc.size());
        for (size_t i = 0; i < acc.size(); ++i) out[i] = rshr_mul128(acc[i], M[i], sh[i]);
        save(dir, "mul128_out", out);
        // the same routine on planted ties and shifts up to 100
        auto acc2 = load<i64>(dir, "mul128x_acc");
        auto M2 = load<u64>(dir, "mul128x_m");
        auto sh2 = load<int32_t>(dir, "mul128x_s");
        std::vector<i64> out2(acc2.size());
        for (size_t i = 0; i < acc2.size(); ++i) out2[i] = rshr_mul128(acc2[i], M2[i], sh2[i]);
        save(dir, "mul128x_out", out2);
    }
    printf("ok\n");
    return 0;
}
