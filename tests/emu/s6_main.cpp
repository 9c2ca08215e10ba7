// Runs the selective-scan kernel's source on the CPU (see cuda_shim.h) on float32 inputs read
// from a file and writes y and h_final (tests/test_s6_kernel_on_cpu.py).
// Input file: int64 B, L, dim, N, G, has_D, has_h0, then float32 x [B][dim][L], delta, A [dim][N],
// B and C [B][G][N][L], D [dim] (if has_D), h0 [B][dim][N] (if has_h0).
// Output file: float32 y [B][dim][L], then h_final [B][dim][N].
#include "cuda_shim.h"
thread_local dim3 threadIdx, blockIdx;
dim3 blockDim, gridDim;
thread_local EmuBlock *emu_block;
#include <cstdio>
#include <vector>
#include "s6_kernel.inc"

template <int NS>
static void run(const std::vector<float> &x, const std::vector<float> &dl, const std::vector<float> &A,
                const std::vector<float> &Bm, const std::vector<float> &Cm, const float *D, const float *h0,
                std::vector<float> &y, std::vector<float> &hf, int64_t B, int64_t L, int64_t dim, int64_t N, int64_t G)
{
    const int cpg = (int)(dim / G);
    const int bpg = (cpg + ssd::kCh - 1) / ssd::kCh;
    emu_launch(dim3((unsigned)(bpg * G), (unsigned)B), dim3(ssd::kThreads), [&] {
        ssd::k_s6_scan<float, float, NS>(x.data(), dl.data(), A.data(), Bm.data(), Cm.data(), D, h0, y.data(),
                                         hf.data(), L, (int)dim, (int)N, (int)G, bpg);
    });
}

int main(int argc, char **argv)
{
    if (argc != 3) return 2;
    FILE *f = std::fopen(argv[1], "rb");
    if (!f) return 3;
    int64_t hdr[7];
    if (std::fread(hdr, sizeof(int64_t), 7, f) != 7) return 4;
    const int64_t B = hdr[0], L = hdr[1], dim = hdr[2], N = hdr[3], G = hdr[4];
    auto rd = [&](size_t n) {
        std::vector<float> v(n);
        if (n && std::fread(v.data(), sizeof(float), n, f) != n) v.clear();
        return v;
    };
    const auto x = rd(B * dim * L), dl = rd(B * dim * L), A = rd(dim * N), Bm = rd(B * G * N * L),
               Cm = rd(B * G * N * L), D = rd(hdr[5] ? dim : 0), h0 = rd(hdr[6] ? B * dim * N : 0);
    std::fclose(f);
    std::vector<float> y(B * dim * L, -999.f), hf(B * dim * N, -999.f);
    const int64_t ns = (N + ssd::kSplit - 1) / ssd::kSplit;
    const float *Dp = hdr[5] ? D.data() : nullptr, *hp = hdr[6] ? h0.data() : nullptr;
    if (ns <= 1) run<1>(x, dl, A, Bm, Cm, Dp, hp, y, hf, B, L, dim, N, G);
    else if (ns <= 2) run<2>(x, dl, A, Bm, Cm, Dp, hp, y, hf, B, L, dim, N, G);
    else if (ns <= 4) run<4>(x, dl, A, Bm, Cm, Dp, hp, y, hf, B, L, dim, N, G);
    else run<8>(x, dl, A, Bm, Cm, Dp, hp, y, hf, B, L, dim, N, G);
    FILE *o = std::fopen(argv[2], "wb");
    if (!o) return 5;
    std::fwrite(y.data(), sizeof(float), y.size(), o);
    std::fwrite(hf.data(), sizeof(float), hf.size(), o);
    std::fclose(o);
    return 0;
}
