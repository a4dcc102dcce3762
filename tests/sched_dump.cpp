// sched_dump.cpp -- prints the tensor-core GEMM's persistent schedule
// (csrc/schedule.h, compiled here as plain C++) for the cases given on
// standard input, one "tiles num_kb resident fix2" line each, so that a test
// can check it without a GPU.  Output per case:
//   case <tiles> <num_kb> <resident> <fix2> <tail_tiles> <tail_clusters> <grid>
//   u <cluster> <i> <tile> <kb0> <kb1> <publish> <others>     (every unit)
#include <cstdio>

#include "schedule.h"

int main() {
    int tiles, num_kb, resident, fix2;
    while (std::scanf("%d %d %d %d", &tiles, &num_kb, &resident, &fix2) == 4) {
        int tt = 0, tc = 0;
        emu::sched_plan_tail(tiles, num_kb, resident, fix2, &tt, &tc);
        const int grid = emu::sched_grid_clusters(tiles, tt, tc, resident);
        std::printf("case %d %d %d %d %d %d %d\n", tiles, num_kb, resident, fix2, tt, tc, grid);
        const emu::TileSchedule s = {tiles, num_kb, tt, tc, grid};
        for (int c = 0; c < grid; ++c) {
            const int n = emu::sched_units(s, c);
            for (int i = 0; i < n; ++i) {
                const emu::Unit w = emu::sched_unit(s, c, i);
                std::printf("u %d %d %d %d %d %d %d\n", c, i, w.tile, w.kb0, w.kb1, w.publish,
                            w.others);
            }
        }
    }
    return 0;
}
