"""Seeded synthetic workloads shared by the tests, the benchmark and the smoke
check.  Input drawing only: no verification arithmetic lives here."""
from .gen import (BF16, F32, Workload, bfs_to_dfs, chain_prefix, chain_tree, config0, config1, config2, config3, config4,
                  expansion_tree_bfs, make_config, random_parent_tree, small_random, tree_kv_rows)
