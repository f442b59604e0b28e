"""Seeded synthetic inputs shared by the tests, the smoke check and the
benchmark.  Input construction only: none of the attention arithmetic."""
