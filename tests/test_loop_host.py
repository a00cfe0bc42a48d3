"""Host logic of the device-resident speculative loop that needs no GPU: the
block-size schedule between listed sizes, chosen from the longest tau of the
last window of rounds."""
import pytest


@pytest.fixture(scope="module")
def next_block_size():
    import __graft_entry__
    __graft_entry__.build()
    from block_diffusion_drafter_layer_gb300.loop import next_block_size as f
    return f


def test_shrinks_to_the_smallest_size_that_covers(next_block_size):
    assert next_block_size([8, 16], 16, 3) == 8
    assert next_block_size([8, 16], 16, 7) == 8     # 8 rows cover tau 7 + 1
    assert next_block_size([8, 16], 16, 8) == 16    # tau 8 + 1 needs more than 8
    assert next_block_size([4, 8, 16], 16, 2) == 4


def test_grows_to_the_largest_once_a_block_is_fully_accepted(next_block_size):
    assert next_block_size([8, 16], 8, 8) == 16
    assert next_block_size([4, 8, 16], 4, 4) == 16  # straight to the largest


def test_keeps_a_size_that_fits(next_block_size):
    assert next_block_size([8, 16], 8, 5) == 8
    assert next_block_size([4, 8, 16], 8, 6) == 8


def test_single_size_never_changes(next_block_size):
    assert next_block_size([16], 16, 1) == 16
    assert next_block_size([16], 16, 16) == 16
