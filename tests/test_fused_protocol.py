"""The fused hc=4 kernel's barrier protocol, model-checked on the CPU under
random interleavings (see fused_protocol_model.py): the kernel's own
configuration never deadlocks or touches a buffer early, and planted protocol
mistakes are caught."""
import pytest

from fused_protocol_model import ProtocolError, simulate


@pytest.mark.parametrize("mixes_only", [False, True])
@pytest.mark.parametrize("stages", [1, 2, 5])
def test_kernel_configuration_runs_clean(stages, mixes_only):
    # 3 ring slots, lag 3, 4 staging buffers: the kernel's constants; 1, 2
    # and 5 stages per tile are d = 1024, 2048 and 5120
    for seed in range(60):
        simulate(ctas=4, tiles=10, stages_per_tile=stages, slots=3, lag=3, bufs=4,
                 mixes_only=mixes_only, seed=seed)


@pytest.mark.parametrize("stages", [1, 3, 5])
def test_post_variant_runs_clean(stages):
    # hc_post of the previous sublayer in front: 8 warps rewrite each stage
    # in place, the MMA waits for all of them, and the MMA thread stores the
    # rewritten stage and releases the slot and the tile's records
    for seed in range(40):
        simulate(ctas=4, tiles=8, stages_per_tile=stages, slots=3, lag=3, bufs=4, post=True,
                 seed=seed)


def test_mma_waiting_for_the_load_instead_of_the_rewrite_is_caught():
    assert _fails(ctas=4, tiles=6, stages_per_tile=2, slots=3, lag=3, bufs=4, post=True,
                  mutation="mma_waits_full")


def test_releasing_a_slot_before_its_store_read_it_is_caught():
    assert _fails(ctas=4, tiles=6, stages_per_tile=2, slots=3, lag=3, bufs=4, post=True,
                  mutation="release_before_store_read")


@pytest.mark.parametrize("stages", [1, 3])
def test_records_before_the_new_stream_is_written_are_caught(stages):
    assert _fails(ctas=4, tiles=6, stages_per_tile=stages, slots=3, lag=3, bufs=4, post=True,
                  mutation="visible_before_written")


@pytest.mark.parametrize("stages", [1, 2, 5])
def test_norm_variant_runs_clean(stages):
    # with the RMSNorm the square warps also send their rows' Gram entries
    # into the owners' records, after the same recv_free wait as the records
    for seed in range(40):
        simulate(ctas=4, tiles=8, stages_per_tile=stages, slots=3, lag=3, bufs=4, norm=True,
                 seed=seed)
    simulate(ctas=16, tiles=4, stages_per_tile=5, slots=3, lag=3, bufs=4, norm=True, seed=1)


def test_gram_entries_sent_without_waiting_for_the_owner_are_caught():
    assert _fails(ctas=4, tiles=6, stages_per_tile=2, slots=3, lag=3, bufs=4, norm=True,
                  mutation="gram_without_recv_free")


def test_full_cluster_of_sixteen():
    for seed in range(3):
        simulate(ctas=16, tiles=4, stages_per_tile=5, slots=3, lag=3, bufs=4, seed=seed)


def test_lag_and_ring_depth_variants_run_clean():
    # the variants timed while tuning the kernel: lags 2 and 4, a 2-slot ring
    for seed in range(10):
        simulate(ctas=4, tiles=8, stages_per_tile=3, slots=3, lag=2, bufs=4, seed=seed)
        simulate(ctas=4, tiles=8, stages_per_tile=3, slots=3, lag=4, bufs=4, seed=seed)
        simulate(ctas=4, tiles=8, stages_per_tile=3, slots=2, lag=3, bufs=4, seed=seed)


def _fails(**kw):
    for seed in range(60):
        try:
            simulate(seed=seed, **kw)
        except ProtocolError:
            return True
    return False


def test_too_few_staging_buffers_for_the_lag_is_caught():
    # two buffers at lag 3: the owner can stage the pre of tile it while the
    # collapse still reads that of tile it-2
    assert _fails(ctas=4, tiles=10, stages_per_tile=2, slots=3, lag=3, bufs=2)


def test_lag_past_the_staging_buffers_is_caught():
    # lag 5 with 4 buffers: a col_done or pre_ready wait can match a phase
    # two rounds away (only the parity is compared)
    assert _fails(ctas=4, tiles=10, stages_per_tile=2, slots=3, lag=5, bufs=4)


def test_releasing_the_records_before_reading_them_is_caught():
    assert _fails(ctas=4, tiles=6, stages_per_tile=2, slots=3, lag=3, bufs=4,
                  mutation="release_before_read")


def test_wrong_empty_slot_parity_is_caught():
    assert _fails(ctas=4, tiles=6, stages_per_tile=2, slots=3, lag=3, bufs=4,
                  mutation="empty_parity")
