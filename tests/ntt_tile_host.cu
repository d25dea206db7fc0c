// ntt_tile_host.cu -- runs the transform numerator's tile arithmetic
// (normalized_cross_correlation_gb300/csrc/ntt_tile.cuh) on the host, pass by
// pass for all 512 thread indices in turn (within a pass the threads touch
// disjoint words, so the order is immaterial), combines the two halves in
// place and reads the correlations back through the column swizzle as the
// kernel does, and writes the centered correlation of every non-wrapping
// shift.  Built and driven by test_ntt_tile_host.py.
//
//   ntt_tile_host wT hT in.bin out.bin [order]
//     in.bin:  256 * 256 tile pixels (uint8, row-major), then hT * wT template
//              pixels (uint8, row-major)
//     order:   0, 1 or 2, the order in which the final combination visits
//              the thread items (see below)
//     out.bin: (257 - hT) * (257 - wT) int32, row-major: for shift (u, v),
//              sum over (j, i) of (tile[u+j][v+i] - 128) * (T[j][i] - 128)
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "../normalized_cross_correlation_gb300/csrc/ntt_tile.cuh"

using namespace ncc::ntt;

int main(int argc, char **argv) {
    if (argc != 5 && argc != 6) {
        std::fprintf(stderr, "usage: %s wT hT in.bin out.bin [order]\n", argv[0]);
        return 2;
    }
    const int wT = std::atoi(argv[1]), hT = std::atoi(argv[2]);
    const int order = argc == 6 ? std::atoi(argv[5]) : 0;
    if (order < 0 || order > 2) return 2;
    if (wT < 1 || hT < 1 || wT > kL || hT > kL) return 2;
    std::vector<uint8_t> img(kL * kL), tmpl((size_t)wT * hT);
    FILE *f = std::fopen(argv[3], "rb");
    if (!f || std::fread(img.data(), 1, img.size(), f) != img.size() ||
        std::fread(tmpl.data(), 1, tmpl.size(), f) != tmpl.size())
        return 3;
    std::fclose(f);

    std::vector<uint32_t> smem(kSmemBytes / 4);
    const Tile t = carve(smem.data());
    for (int tid = 0; tid < kThreads; ++tid) fill_tables(tid, kThreads, t);
    // a pixel's centered value as a residue in [0, p)
    auto pix = [](int v) -> uint32_t { return v >= 128 ? (uint32_t)(v - 128) : (uint32_t)(v - 128 + (int)kP); };
    // the template reversed cyclically: tile entry (a, b) holds T[-a mod 256][-b mod 256]
    auto loadT = [&](int a, int b) -> uint32_t {
        const int j = (kL - a) & (kL - 1), i = (kL - b) & (kL - 1);
        return (j < hT && i < wT) ? pix(tmpl[(size_t)j * wT + i]) : 0u;
    };
    auto loadI = [&](int r, int c) -> uint32_t { return pix(img[(size_t)r * kL + c]); };

    std::vector<uint2> H(2 * kHalf * kL);
    for (int half = 0; half < 2; ++half) {
        for (int tid = 0; tid < kThreads; ++tid)
            half ? rows_fwd1<true>(tid, t, loadT) : rows_fwd1<false>(tid, t, loadT);
        for (int tid = 0; tid < kThreads; ++tid) rows_fwd2(tid, t);
        for (int tid = 0; tid < kThreads; ++tid) cols_fwd1(tid, t);
        for (int tid = 0; tid < kThreads; ++tid) cols_spectrum(tid, t, H.data() + (size_t)half * kHalf * kL);
    }
    // The even half's last pass, per item (the kernel parks it in tensor
    // memory).  Then, as the kernel does: the odd half's last pass combined
    // with it in place -- y[r] = e + w^-r o written back into the buffer
    // words that the same item's last pass read, y[r+128] = e - w^-r o
    // parked -- and each half's correlations read back through the column
    // swizzle.  The items run in the order `order` picks (0: thread-major,
    // 1: item-major, 2: threads in reverse), so any item that read a word
    // another item had already rewritten would change the result.
    std::vector<uint32_t> e((size_t)kThreads * 4 * 16), parked(e.size());
    auto items = [&](auto &&f) {
        if (order == 1) {
            for (int k = 0; k < 4; ++k)
                for (int tid = 0; tid < kThreads; ++tid) f(tid, k);
        } else {
            for (int i = 0; i < kThreads; ++i)
                for (int k = 0; k < 4; ++k) f(order == 2 ? kThreads - 1 - i : i, k);
        }
    };
    for (int half = 0; half < 2; ++half) {
        for (int tid = 0; tid < kThreads; ++tid)
            half ? rows_fwd1<true>(tid, t, loadI) : rows_fwd1<false>(tid, t, loadI);
        for (int tid = 0; tid < kThreads; ++tid) rows_fwd2(tid, t);
        for (int tid = 0; tid < kThreads; ++tid) cols_fwd1(tid, t);
        for (int tid = 0; tid < kThreads; ++tid) cols_mul(tid, t, H.data() + (size_t)half * kHalf * kL);
        for (int tid = 0; tid < kThreads; ++tid) cols_inv(tid, t);
        for (int tid = 0; tid < kThreads; ++tid) rows_inv1(tid, t);
        items([&](int tid, int k) {
            uint32_t out[16];
            rows_inv2(tid, k, t, out);
            const int idx = tid + kThreads * k, r = idx >> 4, n2 = idx & 15;
            if (!half) {
                for (int a = 0; a < 16; ++a) e[(size_t)idx * 16 + a] = out[a];
                return;
            }
            uint32_t *row = t.buf + r * kStride;
            for (int a = 0; a < 16; ++a) {
                const uint32_t ov = mulw(out[a], t.rowFi[r]), ev = red2(e[(size_t)idx * 16 + a]);
                row[16 * a + (n2 ^ a)] = (uint32_t)centered(ev + ov);
                parked[(size_t)idx * 16 + a] = (uint32_t)centered(ev - ov + kP2);
            }
        });
    }
    const int Vy = kL + 1 - hT, Vx = kL + 1 - wT;
    std::vector<int32_t> C((size_t)Vy * Vx);
    auto read_half = [&](int u0) {
        for (int rr = 0; rr < kHalf && u0 + rr < Vy; ++rr)
            for (int xo = 0; xo < Vx; ++xo)
                C[(size_t)(u0 + rr) * Vx + xo] = (int32_t)t.buf[rr * kStride + swz(xo)];
    };
    read_half(0);
    items([&](int tid, int k) {           // the parked half back into the buffer
        const int idx = tid + kThreads * k, r = idx >> 4, n2 = idx & 15;
        for (int a = 0; a < 16; ++a) t.buf[r * kStride + 16 * a + (n2 ^ a)] = parked[(size_t)idx * 16 + a];
    });
    read_half(kHalf);
    f = std::fopen(argv[4], "wb");
    if (!f || std::fwrite(C.data(), 4, C.size(), f) != C.size()) return 4;
    std::fclose(f);
    return 0;
}
