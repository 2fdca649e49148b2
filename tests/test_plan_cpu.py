"""Host-side launch planning of the decode-size kernels (mse_mlp_launch_plan), without a GPU:
the CTA counts the library picks for the gate_up and down launches of a replicated layer or of
a group of ranks, pinned at the shapes whose rules were chosen by measurement, and the rules'
invariants over token counts, tp splits and SM counts."""
import pytest

mse = pytest.importorskip("moe_shared_expert_gb300")

H, I = 7168, 6144   # Kimi-K3 shared expert (hidden, intermediate)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_shared_expert_gb300 import _build
    _build.build()
    mse.lib()


def plan(T, tp=1, rc=1, x_early=False, sm=152):
    return mse.mlp_launch_plan(T, H, I, tp, rc, x_early, sm)


def stream_k_parts(units, kbp, grid):
    """Largest number of CTAs a tile of kbp units is split between when `units` are cut into
    `grid` contiguous equal shares (written from the definition: the owners of a tile's first
    and last unit)."""
    worst = 1
    for t in range(units // kbp):
        first = (t * kbp * grid) // units
        last = ((t * kbp + kbp - 1) * grid) // units
        worst = max(worst, last - first + 1)
    return worst


# -------------------------------------------------------------------- pinned shapes
def test_replicated_decode_layer():
    # gate_up: 96 tiles of 112 k-blocks on 144 CTAs, three CTAs per two tiles (every tile in
    # two parts); the down projection's 56 tiles of 96 k-blocks on 140 CTAs (at most three
    # parts): the largest grids near all SMs with the fewest parts per tile
    for T in (1, 16, 64):
        p = plan(T)
        assert p["swapab"] == 1
        assert (p["gate_up_ctas"], p["gate_up_parts"]) == (144, 2)
        assert (p["down_ctas"], p["down_parts"]) == (140, 3)
        assert p["bn"] == -(-T // 16) * 16 and p["kbs"] == 3


def test_whole_tile_gate_up_from_128_tokens():
    # 128-160 tokens: one CTA per whole gate_up tile (96 CTAs, no split-K finish)
    for T in (128, 144, 160):
        p = plan(T)
        assert (p["gate_up_ctas"], p["gate_up_parts"]) == (96, 1)
        assert p["kbs"] == 2


def test_prefill_kernels_above_160_tokens():
    for T in (161, 192, 256, 300):
        assert plan(T)["swapab"] == 0


@pytest.mark.parametrize("tp,parts", [(8, 8), (16, 16)])
@pytest.mark.parametrize("x_early", [False, True])
def test_one_rank_narrow_slices(tp, parts, x_early):
    # one rank's narrow gate_up slice: every tile in the same number of parts on about two
    # thirds of the SMs (TP8's 12 tiles and TP16's 6 on 96 CTAs); its down projection one CTA
    # per whole tile (56 tiles of 12 / 6 k-blocks), no split-K finish
    p = plan(64, tp, 1, x_early)
    assert (p["gate_up_ctas"], p["gate_up_parts"]) == (96, parts)
    assert (p["down_ctas"], p["down_parts"]) == (56, 1)


def test_tp4_gate_up_beside_the_down_launch_with_early_token_loads():
    # TP4: without early token loads gate_up keeps the stream-K grid; with them it takes the
    # 96 SMs the previous call's 56-CTA down launch leaves free, four parts per tile
    assert (plan(64, 4)["gate_up_ctas"], plan(64, 4)["gate_up_parts"]) == (144, 6)
    p = plan(64, 4, 1, True)
    assert (p["gate_up_ctas"], p["gate_up_parts"]) == (96, 4)
    assert p["down_ctas"] == 56 and p["gate_up_ctas"] + p["down_ctas"] == 152


def test_tuning_overrides():
    old = mse.set_tuning(mse.TUNE_GRID_DOWN, 128)
    try:
        p = plan(64)
        assert p["down_ctas"] == 128 and p["gate_up_ctas"] == 144
        assert p["down_parts"] == stream_k_parts(56 * 96, 96, 128)
    finally:
        mse.set_tuning(mse.TUNE_GRID_DOWN, old)
    old = mse.set_tuning(mse.TUNE_GRID, 120)
    try:
        p = plan(64)
        assert p["gate_up_ctas"] == 120 and p["down_ctas"] == 120   # GRID_DOWN 0: as GRID
        p = plan(64, 8, 1, True)   # a set grid also turns off the narrow and co-resident rules
        assert p["gate_up_ctas"] == 120 and p["down_ctas"] == 120
    finally:
        mse.set_tuning(mse.TUNE_GRID, old)
    old = mse.set_tuning(mse.TUNE_ISSUE_GROUP, 2)
    try:
        assert plan(64)["kbs"] == 2
    finally:
        mse.set_tuning(mse.TUNE_ISSUE_GROUP, old)
    assert plan(64) == plan(64, sm=152)   # everything restored


# -------------------------------------------------------------------- invariants
@pytest.mark.parametrize("sm", [152, 148, 132, 100, 80])
def test_plan_invariants(sm):
    cap = min(sm, 160)
    for T in (1, 7, 16, 33, 64, 100, 128, 160):
        for tp in (1, 2, 4, 8, 16):
            for rc in sorted({1, tp // 2 or 1, tp}):
                for xe in (False, True):
                    p = plan(T, tp, rc, xe, sm)
                    assert p["swapab"] == 1, (T, tp, rc, xe, sm)
                    sw = I // tp
                    n_gt, kbp_gu = rc * sw // 64, H // 64
                    n_dn, kbp_dn = rc * (H // 128), sw // 64
                    gu, dn = p["gate_up_ctas"], p["down_ctas"]
                    assert 1 <= gu <= min(cap, n_gt * kbp_gu) and 1 <= dn <= min(cap, n_dn * kbp_dn)
                    # the reported parts are those of a stream-K cut of the units over the grid
                    assert p["gate_up_parts"] == stream_k_parts(n_gt * kbp_gu, kbp_gu, gu)
                    assert p["down_parts"] == stream_k_parts(n_dn * kbp_dn, kbp_dn, dn)
                    assert p["bn"] == -(-T // 16) * 16 and 1 <= p["kbs"] <= 4 and p["stages"] >= 2
                    # narrow down projections (at most 24 k-blocks per tile) run whole tiles
                    # whenever every tile has an SM
                    if kbp_dn <= 24 and n_dn <= cap:
                        assert (dn, p["down_parts"]) == (n_dn, 1)
                    # with early token loads a gate_up grid that differs from the grid without
                    # them fits beside the down launch, every tile in the same number of parts
                    q = plan(T, tp, rc, False, sm)
                    if xe and gu != q["gate_up_ctas"]:
                        assert gu + dn <= cap and gu % n_gt == 0
                        assert p["gate_up_parts"] == gu // n_gt


def test_plan_errors_and_unsupported_options():
    out_of_range = [(0, H, I, 1, 1), (64, H, I, 8, 9), (64, H, I, 0, 1), (64, H, I, 8, 0)]
    for T_, H_, I_, tp, rc in out_of_range:
        with pytest.raises(mse.MSEError):
            mse.mlp_launch_plan(T_, H_, I_, tp, rc)
    with pytest.raises(mse.MSEError):
        mse.mlp_launch_plan(64, H, 6000, 7)          # I not divisible by tp
    with pytest.raises(mse.MSEError):
        mse.mlp_launch_plan(64, H, I, sm_count=0)
    # shapes off the 64-column grid, or the generic path forced, take the generic kernels
    assert mse.mlp_launch_plan(64, 7200, I)["swapab"] == 0
    old = mse.set_kernel_path(mse.PATH_GENERIC)
    try:
        assert plan(64)["swapab"] == 0
    finally:
        mse.set_kernel_path(old)
    for key in (mse.TUNE_ONE_LAUNCH, mse.TUNE_PAIR_MIN_T, mse.TUNE_CLUSTER_FINISH):
        old = mse.set_tuning(key, 1)
        try:
            with pytest.raises(mse.MSEError):
                plan(64)
        finally:
            mse.set_tuning(key, old)
    assert plan(64)["swapab"] == 1


# -------------------------------------------------------------------- merged projection
Q, KV, TP16 = 1536, 576, 16   # q_a and kv_a rows of the merged projection, TP16 layout


def test_merged_projection_aligned_grid():
    # 17 weight tiles of 128 rows (2112 rows) and 112 k-blocks: every grid near all SMs splits
    # some tile more than three ways, so the launch takes the grid that puts every tile in the
    # same number of parts (136 CTAs, 8 parts each), finished jointly
    for T in (1, 64, 128, 160):
        p = mse.merged_launch_plan(T, H, Q, KV, TP16)
        assert (p["swapab"], p["ctas"], p["parts"], p["joint_finish"]) == (1, 136, 8, 1)
        assert p["bn"] == -(-T // 16) * 16


@pytest.mark.parametrize("sm", range(40, 161, 7))
def test_merged_projection_grid_rule_over_sm_counts(sm):
    p = mse.merged_launch_plan(128, H, Q, KV, TP16, sm)
    g_max, n_tiles, kbp = min(sm, 160), 17, H // 64
    assert p["parts"] == stream_k_parts(n_tiles * kbp, kbp, p["ctas"])
    per = g_max // n_tiles
    if p["ctas"] != g_max:
        # the aligned grid: a multiple of the tile count, at least 80% of the SMs
        assert p["ctas"] == n_tiles * per and 5 * p["ctas"] >= 4 * g_max and p["parts"] == per
    assert p["joint_finish"] == (1 if p["parts"] >= 6 else 0)


def test_merged_plan_errors():
    with pytest.raises(mse.MSEError):
        mse.merged_launch_plan(128, H, 1536, 577, 16)   # kv_dim not divisible by tp
    with pytest.raises(mse.MSEError):
        mse.merged_launch_plan(0, H, Q, KV, TP16)
    assert mse.merged_launch_plan(300, H, Q, KV, TP16)["swapab"] == 0   # the prefill kernels
    assert mse.merged_launch_plan(128, 7200, Q, KV, TP16)["swapab"] == 0   # the generic kernels
