// Host check of the chunk-slot arithmetic of packed_seq.cuh (the layout the KDA backward and the
// DPLR kernels index their workspaces by): for random packings, every chunk of every sequence
// maps to a slot inside the workspace, no two chunks share a slot (chunk or state), and the
// bisection of a packed CTA finds the sequence and chunk that own its slot.  Offsets outside
// [0, T] and decreasing ones (clamped by the kernels) must stay inside the workspace.
// Exit status 0 when every check holds; the first failure is printed.
#include <cstdio>
#include <cstdlib>
#include <set>
#include <vector>

#include "packed_seq.cuh"

struct Params {
    int B, T;
    const int *cu_seqlens;
};

template <int C>
static int check(const Params &p, bool monotone, int H) {
    using namespace kda::seq;
    const bool packed = p.cu_seqlens != nullptr;
    const int NS = chunk_slots<C>(p.B, p.T, packed);
    std::set<size_t> cslots, sslots;
    for (int b = 0; b < p.B; ++b) {
        const Seq sq = seq_of<C>(p, b);
        if (sq.row0 < 0 || sq.len < 0 || sq.row0 + sq.len > (packed ? p.T : p.B * p.T)) return 1;
        for (int h = 0; h < H; ++h) {
            for (int n = 0; n < sq.nch; ++n) {
                const size_t ci = chunk_index<C>(p, sq, h, n);
                if (ci >= (size_t)H * NS) return 2;
                if (monotone && !cslots.insert(ci).second) return 3;
                const int t0 = n * C, nvalid = sq.len - t0 < C ? sq.len - t0 : C;
                if (nvalid < 1) return 4;
            }
            for (int n = 0; n <= sq.nch; ++n) {
                const size_t si = state_index<C>(p, sq, b, h, n);
                if (si >= (size_t)H * (NS + p.B)) return 5;
                if (monotone && !sslots.insert(si).second) return 6;
            }
        }
    }
    if (packed) {
        for (int s = 0; s < NS; ++s) {
            int b, n;
            Seq sq;
            const bool used = slot_of<C>(p, s, b, n, sq);
            if (b < 0 || b >= p.B) return 7;
            if (used && (n < 0 || n >= sq.nch || sq.slot0 + n != s)) return 8;
            if (monotone && used != (cslots.count((size_t)s) == 1)) return 9;
        }
    }
    return 0;
}

int main() {
    srand(12345);
    for (int trial = 0; trial < 4000; ++trial) {
        const int B = 1 + rand() % 9;
        const bool monotone = rand() % 5 != 0;
        std::vector<int> cu(B + 1);
        int T;
        if (monotone) {
            cu[0] = 0;
            for (int b = 0; b < B; ++b) {
                const int pick[6] = {0, 1, 15, 16, 17, rand() % 160};
                cu[b + 1] = cu[b] + pick[rand() % 6];
            }
            T = cu[B] > 0 ? cu[B] : 1;
        } else {
            T = 1 + rand() % 300;
            for (int b = 0; b <= B; ++b) cu[b] = rand() % (T + 100) - 50;
        }
        const int H = 1 + rand() % 3;
        const Params packed{B, T, cu.data()}, dense{B, T, nullptr};
        const int r = check<16>(packed, monotone, H) * 100 + check<32>(packed, monotone, H) * 10 +
                      check<64>(dense, true, H);
        if (r) {
            std::printf("trial %d: B %d T %d monotone %d: failure code %d\n", trial, B, T, (int)monotone, r);
            return 1;
        }
    }
    std::printf("ok\n");
    return 0;
}
