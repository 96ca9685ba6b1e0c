"""CPU oracle for the ragged batched speculative-verify step.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
bench's CPU-baseline leg; never by the product library or its binding.
"""
